// Absorbed-branch MLA verify on GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// "One guard, 110x off the verify step", section "The defect": fold the key
// up-projection into the query, attend against the compressed latent, then
// apply the value up-projection.  Three kernels (the GEMM runs twice), all
// bf16 operands with fp32 accumulation in tensor memory:
//
//  swapab_gemm     fold: q_lat[row, h, :] = q_nope[row, h, :] . W_UK[h] (n -> 512)
//                  and unembed: out[row, h, :] = o_lat[row, h, :] . W_UV[h]
//                  (512 -> v).  Swap-AB GEMM per head: D[M x rows] = W[h]^T x
//                  act^T, so the weight is the 128-row operand read once for
//                  all B*L rows (the pages' "small-M verify" idea, "Draft caps
//                  and calibration", section "Small-M verify kernel").
//  absorbed_attn   split-KV attention of the L*H query rows of a sequence
//                  against [c_kv || k_rope] (576 wide), online softmax, causal
//                  verify mask, o_lat = P . c_kv accumulated in the latent space.
//                  Each latent tile is read once for all 128 rows of a tile
//                  ("Multi-row attention kernel" on the same page).  A cluster
//                  of two CTAs shares one 128-row tile: CTA j holds latent
//                  columns [256j, 256j+256) and RoPE columns [32j, 32j+32),
//                  computes its partial scores over its columns, swaps them
//                  with the peer through distributed shared memory, and both
//                  accumulate their half of o_lat (128 x 256 fp32 in TMEM).
//  unembed_merge   the split-KV merge and the unembedding in one kernel: they
//                  commute, so every piece's rows are multiplied by W_UV in one
//                  TMA-fed tensor-core GEMM and the products are combined with
//                  the pieces' log-sum-exp weights (see the kernel).  When a
//                  sequence has more than 64 pieces, merge_sm103 /
//                  merge_rows_sm103 (log-sum-exp merge into bf16 o_lat) and the
//                  swap-AB unembedding run instead.
//
// The launches are chained with programmatic dependent launch: each one
// starts the loads that do not depend on its predecessor (weights, the KV
// cache) before waiting for it.
//
// Every wait is bounded; a wait that runs out sets the status word and the
// kernel finishes without waiting further (results are then undefined and
// mla_device_status reports MLA_ERR_TIMEOUT).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <cmath>
#include <mutex>
#include <utility>

#include "mla_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace mla {
using namespace sm103;

static __device__ int g_absorbed_status;

namespace {

constexpr int kLat = 512;

// The first 1024-byte boundary at or after the dynamic shared array, as an
// offset from the array itself (no integer round trip), so that the compiler
// still knows every pointer derived from it is a shared-memory one.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (sm103::smem_u32(p) & 1023u)) & 1023u);
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
// swap-AB small-M GEMM (fold and unembed)
// =========================================================================
// out[row, h, m] = sum_k act[row, h, k] * W[h][k][m] for the B*L rows of a call:
//   fold:    act = q_nope (K = n),    W = W_UK [H, n, 512], out = q_lat (M = 512)
//   unembed: act = o_lat  (K = 512),  W = W_UV [H, 512, v], out = out   (M = v)
// One CTA per (128-wide M tile, head, block of NB rows): D[128 x NB] =
// W[h][:, tile]^T (MN-major, the 128-row operand) x act^T (K-major).  The
// weight is read once for all rows.  K arrives in 64-wide chunks, each with
// its own barrier, and each chunk's MMAs issue as soon as it lands.
struct GemmParams {
  __nv_bfloat16* out;  // [rows, H, M], or the attention's Q tiles (see below)
  int rows, H, K, M, NB;
  // L > 0: write q_lat as the attention reads it.  Query row r = l*H + h of
  // sequence b belongs to tile r/128 (row r%128 in it); a tile is 64 chunks of
  // 8 latent columns, each chunk 128 rows x 16 B, so a warp that loads one
  // chunk for its 32 rows reads 512 contiguous bytes.
  int L, ntile;
};

constexpr int GEMM_MAX_K = 512;

__global__ void __launch_bounds__(128) swapab_gemm_sm103(const __grid_constant__ CUtensorMap tm_w,
                                                         const __grid_constant__ CUtensorMap tm_act,
                                                         GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int mt = blockIdx.x, h = blockIdx.y, row0 = blockIdx.z * p.NB;
  const int K = p.K, nk = K / 64, NB = p.NB;
  uint8_t* sA = smem;                    // 2 atoms x K rows x 128 B
  uint8_t* sB = smem + 2 * K * 128;      // nk chunks x NB rows x 128 B
  uint64_t* bars = (uint64_t*)(sB + nk * NB * 128);   // [0, nk): chunk k landed; nk: MMA done
  uint32_t* slot = (uint32_t*)(bars + GEMM_MAX_K / 64 + 1);
  volatile int* fail = (volatile int*)(slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = tmem_cols_for(NB);

  if (threadIdx.x == 0) {
    for (int k = 0; k <= nk; ++k) mbar_init(smem_u32(&bars[k]), 1);
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
    // the weights do not depend on the preceding kernel: start them first
    for (int kc = 0; kc < nk; ++kc) {
      const uint32_t bk = smem_u32(&bars[kc]);
      mbar_arrive_expect_tx(bk, 2 * 64 * 128 + NB * 128);
      for (int j = 0; j < 2; ++j)
        tma_load_2d(smem_u32(sA + j * K * 128 + kc * 8192), &tm_w, bk, mt * 128 + 64 * j,
                    h * K + 64 * kc);
    }
    pdl_wait();  // the activations may come from the preceding kernel
    // The next kernel may launch now and start its own independent loads (it
    // waits for this grid before reading what this one writes).  Triggering
    // only after this grid's own wait means a kernel that follows starts
    // after the kernel before this one has finished, so what that kernel
    // wrote (lengths, page table, index lists) is complete for it.
    pdl_launch_dependents();
    for (int kc = 0; kc < nk; ++kc)
      tma_load_2d(smem_u32(sB + kc * NB * 128), &tm_act, smem_u32(&bars[kc]), h * K + 64 * kc,
                  row0);
    const uint32_t idesc = idesc_bf16(128, NB, 1, 0);
    for (int kc = 0; kc < nk && ok; ++kc) {
      wait_or_fail(ok, smem_u32(&bars[kc]), 0, 1);
      if (!ok) break;
      tc_fence_after();
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem, sdesc_sw128(smem_u32(sA) + (kc * 64 + ks * 16) * 128, K * 128, 1024),
                 sdesc_sw128(smem_u32(sB) + kc * NB * 128 + ks * 32, 16, 1024), idesc,
                 (kc | ks) != 0);
    }
    if (ok) {
      mma_commit(smem_u32(&bars[nk]));
      wait_or_fail(ok, smem_u32(&bars[nk]), 0, 2);
    }
    if (!ok) *fail = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (!*fail) {
    // D[m][row] leaves through the drained weight buffer, 64 rows at a time:
    // staged as bf16 [row][128 columns] (16-byte chunks XOR-swizzled by row),
    // then written as 16-byte chunks of 8 consecutive output columns.
    uint8_t* stg = sA;  // 64 rows x 256 B (the weight buffer holds at least 16 KB)
    const int ml = warp * 32 + lane;  // this thread's TMEM lane = column of the tile
    for (int g0 = 0; g0 < NB; g0 += 64) {
      const int gn = min(64, NB - g0);
      for (int c0 = 0; c0 < gn; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + g0 + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int rl = c0 + i;
          *(__nv_bfloat16*)(stg + rl * 256 + ((((ml >> 3) ^ (rl & 15))) << 4) + (ml & 7) * 2) =
              __float2bfloat16_rn(__uint_as_float(v[i]));
        }
      }
      __syncthreads();
      for (int k = threadIdx.x; k < gn * 16; k += 128) {
        // q_lat tiles: a column chunk's rows are contiguous, so consecutive
        // threads take consecutive rows; row-major output: consecutive chunks
        int rl, mc;
        if (p.L > 0) {
          mc = k / gn;
          rl = k - mc * gn;
        } else {
          rl = k >> 4;
          mc = k & 15;
        }
        const int row = row0 + g0 + rl;
        if (row >= p.rows) continue;
        const uint4 val = *(const uint4*)(stg + rl * 256 + ((mc ^ (rl & 15)) << 4));
        const int m = mt * 128 + mc * 8;
        size_t idx;
        if (p.L > 0) {
          const int b = row / p.L, r = (row - b * p.L) * p.H + h;
          idx = ((((size_t)b * p.ntile + (r >> 7)) * 64 + (m >> 3)) * 128 + (r & 127)) * 8;
        } else {
          idx = ((size_t)row * p.H + h) * p.M + m;
        }
        *(uint4*)(p.out + idx) = val;
      }
      __syncthreads();
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
constexpr int STAGES = 4;
constexpr int NWG = 2;                  // softmax warpgroups; each takes 1/NWG of a row
constexpr int CPT = 64 / NWG;           // score columns per softmax thread
constexpr int OPT = 256 / NWG;          // O (and latent Q) columns per softmax thread
constexpr int SOFTMAX_THREADS = 128 * NWG;
constexpr int XCHG_WARP0 = 3 + SOFTMAX_THREADS / 32;  // first of the four score-exchange warps
// producer, S issuer, P.V issuer, softmax, score exchange
constexpr int ATTN_THREADS = 96 + SOFTMAX_THREADS + 128;
constexpr int Q_ROPE = BM * 64;         // the 32 RoPE columns of this CTA's Q rows (64-B swizzle)
constexpr int KV_CHUNK = BN * 128;      // one 64-column bf16 chunk of a KV tile
constexpr int KV_ROPE = BN * 64;        // 32 RoPE columns of a KV tile
constexpr int P_TILE = BM * 128;        // one bf16 P tile (128 rows x 64 positions)
constexpr int X_BYTES = BM * BN * 2;    // partial scores of a tile, fp16 [128][64]
constexpr int OFF_QR = 0;
constexpr int OFF_KV = OFF_QR + Q_ROPE;
constexpr int KV_STAGE = 4 * KV_CHUNK + KV_ROPE;
constexpr int OFF_P = OFF_KV + STAGES * KV_STAGE;   // the P tile
constexpr int OFF_X = OFF_P + P_TILE;               // the peer's partial scores land here (x2)
constexpr int OFF_STG = OFF_X + 2 * X_BYTES;        // this CTA's partial scores, outgoing
constexpr int OFF_RED = OFF_STG + X_BYTES;          // row maxima of the warpgroups
constexpr int OFF_LS = OFF_RED + NWG * BM * 4;      // row sums of the warpgroups
constexpr int OFF_BAR = OFF_LS + NWG * BM * 4;
constexpr int ATTN_SMEM = OFF_BAR + 256 + 1024;     // + barriers + alignment slack
// Tensor memory: O half [0,256) fp32; this CTA's 256 latent query columns as
// bf16 pairs [256,384) (the A operand of the score MMAs); S buffers [384,512).
constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_QL = 256;
constexpr uint32_t TM_S = 384;
constexpr int SBUF = 2;
static_assert(OFF_KV % 1024 == 0 && KV_STAGE % 1024 == 0 && OFF_P % 1024 == 0,
              "swizzle atoms need 1 KiB alignment");
static_assert(ATTN_SMEM <= 232448, "shared memory per CTA");

struct AttnParams {
  const int32_t* lens;
  const int32_t* page_table;
  const __nv_bfloat16* q_lat;  // Q tiles [B, rtiles, 64 chunks, 128 rows, 8] bf16
  int page_size, max_pages, num_pages;
  long long seq_stride;
  int L, H, R;        // R = L*H query rows per sequence
  int rtiles;         // ceil(R / 128)
  int B;
  int chunk, splits;  // KV rows per split (multiple of 64), splits per sequence (max)
  float sl2;          // softmax scale * log2(e)
  __nv_bfloat16* o_part;  // [B, splits, R, 512]: O / l of each piece
  float* ml;              // [B, splits, R, 2]: (m, l) of each piece
  const char* pf;     // W_UV, pulled into L2 while the attention runs
  size_t pf_bytes;
  // index-list (top-k) mode: [B, L, topk_k] positions per verify row, and the
  // cache as plain pointers (rows are gathered one by one)
  const int32_t* topk;
  int topk_k;
  const char* ckv;
  const char* kr;
  long long ckv_stride, kr_stride;  // elements between rows
};

// Barrier slots.  Every barrier that is waited on by parity alone has enough
// copies that it cannot complete twice before its waiter looks.
enum {
  B_QFULL = 0, B_QTMEM = 1, B_KVFULL = 2, B_KVEMPTY = 6, B_SFULL = 10, B_SFREE = 12,
  B_PFULL = 14, B_ODONE = 16, B_XFULL = 18, B_XFREE = 20, B_DRAIN = 22, B_COUNT = 24
};

// One partial score of this CTA in log2-softmax units, rounded to fp16: the
// exchange warps send exactly this to the peer and the softmax adds exactly
// this to the peer's, so both CTAs of a pair sum the same two rounded values
// and their scores agree bit for bit.  (Packed conversions: the scalar ones
// would crowd the pipe the exponentials need.)
__device__ __forceinline__ __half2 round_partial(uint32_t a, uint32_t b, float sl2) {
  return __floats2half2_rn(__uint_as_float(a) * sl2, __uint_as_float(b) * sl2);
}

// This thread's CPT partial scores of tile j (columns c0..c0+CPT-1 of this
// CTA's share) from TMEM, rounded as they are sent, in fp32.
__device__ __forceinline__ void load_partial(bool& ok, uint32_t tmem, uint32_t lane_base, int c0,
                                             int j, uint32_t bar_sfull0, uint32_t bar_sfree0,
                                             float sl2, float (&s)[CPT]) {
  const int sb = j & (SBUF - 1);
  wait_or_fail(ok, bar_sfull0 + 8 * sb, (j / SBUF) & 1, 20);
  tc_fence_after();
  uint32_t v[CPT];
#pragma unroll
  for (int k = 0; k < CPT / 16; ++k)
    tmem_ld16(tmem + lane_base + TM_S + sb * BN + c0 + 16 * k, *(uint32_t(*)[16])(v + 16 * k));
  tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < CPT / 2; ++e) {
    const float2 f = __half22float2(round_partial(v[2 * e], v[2 * e + 1], sl2));
    s[2 * e] = f.x;
    s[2 * e + 1] = f.y;
  }
  tc_fence_before();
  mbar_arrive(bar_sfree0 + 8 * sb);
}

// Exchange tile layout: [lane quarter][warpgroup][32 rows][2*CPT B] (a row's
// CPT fp16 partial scores of that warpgroup's columns), 16-byte chunks
// XOR-swizzled by row so a warp's accesses hit distinct banks.  The 32 rows of
// one TMEM lane quarter are one contiguous block, which one exchange warp
// ships to the peer with a single bulk copy.
constexpr int XROW = 2 * CPT;                   // bytes per row and warpgroup
constexpr int XCH = XROW / 16;                  // 16-byte chunks per row and warpgroup
constexpr int XQUARTER = 32 * XROW * NWG;       // bytes per lane quarter
__device__ __forceinline__ uint32_t xchg_offset(int wg, int q, int c) {
  const int sw = XCH == 4 ? ((q >> 1) & 3) : XCH == 2 ? ((q >> 2) & 1) : 0;
  return (uint32_t)((q >> 5) * XQUARTER + wg * (32 * XROW) + (q & 31) * XROW + ((c ^ sw) << 4));
}

// SPARSE: the index-list mode ("One guard, 110x off the verify step", section
// "The sparse model is different": attention runs over the cached positions
// an indexer selected).  A tile's 64 columns are list entries j of its verify
// row (all rows of a 128-row tile belong to one verify row: H is a multiple
// of 128); the producer warp gathers their cache rows with 16-byte cp.async
// copies into the layout the TMA boxes would give, zero-filling entries that
// are padding (< 0), past the row's causal limit or on a bad page, and the
// softmax masks those columns.  Pieces split the list instead of [0, T).
template <bool SPARSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(ATTN_THREADS, 1)
    absorbed_attn_sm103(const __grid_constant__ CUtensorMap tm_qr,
                        const __grid_constant__ CUtensorMap tm_ckv,
                        const __grid_constant__ CUtensorMap tm_kr,
                        const __grid_constant__ CUtensorMap tm_op, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int tile = blockIdx.x >> 1, split = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // (the sequence length is first needed after the barrier and TMEM setup
  // below, which its load overlaps)
  const int T = p.lens[b];

  uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
  uint32_t* slot = (uint32_t*)(bars + B_COUNT + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQR = smem_u32(smem + OFF_QR), sKV = smem_u32(smem + OFF_KV);
  const uint32_t sP = smem_u32(smem + OFF_P), sX = smem_u32(smem + OFF_X);
  const uint32_t sStg = smem_u32(smem + OFF_STG);
  float* red = (float*)(smem + OFF_RED);
  float* lsum = (float*)(smem + OFF_LS);

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QTMEM), SOFTMAX_THREADS);
    for (int s = 0; s < STAGES; ++s) {
      // index-list mode: each producer lane's copies arrive on their own
      mbar_init(bar(B_KVFULL + s), SPARSE ? 32 : 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SFREE + s), SOFTMAX_THREADS + 4);  // + one per exchange warp
      mbar_init(bar(B_PFULL + s), SOFTMAX_THREADS);
      mbar_init(bar(B_ODONE + s), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_XFULL + k), 1);
      mbar_init(bar(B_XFREE + k), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int klen = SPARSE ? p.topk_k : T;  // list entries, or positions
  const int nsplit = (klen + p.chunk - 1) / p.chunk;
  if (split >= nsplit) {  // both CTAs of the cluster leave together, the peer untouched
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }
  const int row0 = tile * BM;
  const int l_last = min(p.R - 1, row0 + BM - 1) / p.H;
  const int vis_end = T - p.L + l_last + 1;
  const int kv0 = split * p.chunk;
  const int kv1 = SPARSE ? min(kv0 + p.chunk, klen) : min(min(kv0 + p.chunk, T), vis_end);
  const int ntiles = kv1 > kv0 ? (kv1 - kv0 + BN - 1) / BN : 0;
  // arm the exchange barriers for tiles 0 and 1 (the peer's bulk copies count
  // them down), then publish the setup to the peer: each role waits for the
  // peer's setup only before its first access to the peer, so the KV loads,
  // the query load and the score MMAs do not wait for the slower CTA
  if (threadIdx.x == 0) {
    if (ntiles > 0) mbar_arrive_expect_tx(bar(B_XFULL), X_BYTES);
    if (ntiles > 1) mbar_arrive_expect_tx(bar(B_XFULL + 1), X_BYTES);
  }
  cluster_arrive();
  pdl_launch_dependents();  // the merge may launch; it waits for this grid

  if (warp == 0 && SPARSE) {
    // ------------------------------------------- gathering producer (32 lanes)
    if (ntiles > 0) {
      bool ok = true;
      pdl_wait();  // the index list may come from the preceding kernel
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_QFULL), Q_ROPE);
        tma_load_2d(sQR, &tm_qr, bar(B_QFULL), (int)rank * 32, b * p.R + row0);
      }
      const int l = row0 / p.H;
      const int last_t = T - p.L + l;
      const int32_t* list = p.topk + ((size_t)b * p.L + l) * p.topk_k;
      // list entry of row lane + 32 u of tile i, or -1 past the piece
      auto entry = [&](int i, int u) -> int {
        const int j = kv0 + i * BN + lane + 32 * u;
        return (i < ntiles && j < kv1) ? list[j] : -1;
      };
      // the entries of the next four tiles are loaded ahead of their copies
      // (in rotating registers), so a tile's rows are known when its turn comes
      int e0a = entry(0, 0), e0b = entry(0, 1), e1a = entry(1, 0), e1b = entry(1, 1);
      int e2a = entry(2, 0), e2b = entry(2, 1), e3a = entry(3, 0), e3b = entry(3, 1);
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % STAGES;
        const int ta = e0a, tb = e0b;
        e0a = e1a;
        e0b = e1b;
        e1a = e2a;
        e1b = e2b;
        e2a = e3a;
        e2b = e3b;
        e3a = entry(i + 4, 0);
        e3b = entry(i + 4, 1);
        if (i >= STAGES) {
          if (lane == 0) wait_or_fail(ok, bar(B_KVEMPTY + s), ((i / STAGES) - 1) & 1, 10);
          ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
          if (!ok) break;
        }
        // this lane resolves tile rows lane and lane + 32: the cache row of
        // the listed position, or -1 (zero-filled, masked)
        long long crow[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int t = u == 0 ? ta : tb;
          crow[u] = -1;
          if (t >= 0 && t <= last_t) {
            if (p.page_table) {
              const int page = p.page_table[(long long)b * p.max_pages + t / p.page_size];
              if (page < 0 || page >= p.num_pages) report_timeout(kBadPageSite);
              else crow[u] = (long long)page * p.page_size + (t % p.page_size);
            } else {
              crow[u] = (long long)b * p.seq_stride + t;
            }
          }
        }
        const uint32_t st = sKV + s * KV_STAGE;
        // latent: this CTA's 256 columns of a row are 512 bytes, one 16-byte
        // chunk per lane; chunk c of row jr lands where the 128-byte-swizzled
        // box of its 64 columns puts it
        for (int jr = 0; jr < BN; ++jr) {
          const long long cr = __shfl_sync(0xffffffffu, crow[jr >> 5], jr & 31);
          const uint32_t dst =
              st + (lane >> 3) * KV_CHUNK + jr * 128 + ((((lane & 7) ^ (jr & 7))) << 4);
          const char* src = cr >= 0 ? p.ckv + (cr * p.ckv_stride + 256 * rank) * 2 + lane * 16
                                    : p.ckv;
          cp_async16(dst, src, cr >= 0 ? 16u : 0u);
        }
        // RoPE: 32 columns (64 bytes, 64-byte swizzle) per row, 8 rows per round
        for (int jr0 = 0; jr0 < BN; jr0 += 8) {
          const int jr = jr0 + (lane >> 2), c = lane & 3;
          const long long cr = __shfl_sync(0xffffffffu, crow[jr0 >> 5], jr & 31);
          const uint32_t dst = st + 4 * KV_CHUNK + jr * 64 + ((c ^ ((jr >> 1) & 3)) << 4);
          const char* src =
              cr >= 0 ? p.kr + (cr * p.kr_stride + 32 * rank) * 2 + c * 16 : p.kr;
          cp_async16(dst, src, cr >= 0 ? 16u : 0u);
        }
        cp_async_mbar_arrive(bar(B_KVFULL + s));
      }
      // nothing this warp started may still be landing when the CTA exits
      cp_async_wait_all();
      if (lane == 0) mbar_wait(bar(B_QFULL), 0);
    }
    cluster_wait();  // (this role never touches the peer)
    cluster_arrive();  // done with the peer: the exit barrier's arrival
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      prefetch_tmap(&tm_ckv);
      const int qrow = b * p.R + row0;
      auto load_kv = [&](int i) {
        const int s = i % STAGES;
        const int t0 = kv0 + i * BN;
        long long y;
        if (p.page_table) {
          const int page = p.page_table[(long long)b * p.max_pages + t0 / p.page_size];
          // an id outside [0, num_pages) forms no address: the box is read
          // from wholly negative rows, which TMA fills with zeros
          if (page < 0 || page >= p.num_pages) {
            report_timeout(kBadPageSite);
            y = -2 * BN;
          } else {
            y = (long long)page * p.page_size + (t0 % p.page_size);
          }
        } else {
          y = (long long)b * p.seq_stride + t0;
        }
        const uint32_t st = sKV + s * KV_STAGE;
        mbar_arrive_expect_tx(bar(B_KVFULL + s), KV_STAGE);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(st + c * KV_CHUNK, &tm_ckv, bar(B_KVFULL + s), (int)(4 * rank + c) * 64,
                      (int)y);
        tma_load_2d(st + 4 * KV_CHUNK, &tm_kr, bar(B_KVFULL + s), (int)rank * 32, (int)y);
      };
      // the cache does not depend on the preceding kernel: start every stage now
      const int pre = min(ntiles, STAGES);
      for (int i = 0; i < pre; ++i) load_kv(i);
      // q_rope is a call input; it still waits so no read overtakes the predecessor
      pdl_wait();
      mbar_arrive_expect_tx(bar(B_QFULL), Q_ROPE);
      tma_load_2d(sQR, &tm_qr, bar(B_QFULL), (int)rank * 32, qrow);
      // The unembedding weights are read right after this kernel; at verify
      // widths the attention leaves HBM mostly idle, so each CTA pulls a slice
      // into L2 -- once its own first KV tiles have landed, so that the two do
      // not share the HBM bandwidth the first tiles wait for.
      if (p.pf != nullptr) {
        mbar_wait(bar(B_KVFULL + (pre - 1) % STAGES), 0);
        const size_t nct = (size_t)gridDim.x * gridDim.y * gridDim.z;
        const size_t id = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        const size_t slice = ((p.pf_bytes + nct - 1) / nct + 4095) & ~(size_t)4095;
        for (size_t o = id * slice; o < min(p.pf_bytes, (id + 1) * slice); o += 32768)
          prefetch_l2(p.pf + o, (uint32_t)min((size_t)32768, p.pf_bytes - o));
      }
      int issued = pre;
      for (int i = STAGES; i < ntiles; ++i) {
        wait_or_fail(ok, bar(B_KVEMPTY + i % STAGES), ((i / STAGES) - 1) & 1, 10);
        if (!ok) break;
        load_kv(i);
        issued = i + 1;
      }
      // nothing this thread started may still be landing when the CTA exits
      mbar_wait(bar(B_QFULL), 0);
      for (int i = max(issued - STAGES, 0); i < issued; ++i)
        mbar_wait(bar(B_KVFULL + i % STAGES), (i / STAGES) & 1);
    }
    cluster_wait();  // (this role never touches the peer)
    cluster_arrive();  // done with the peer: the exit barrier's arrival
  } else if (warp == 1) {
    // ------------------------------------------------------- score-MMA issuer
    // S(i) = Q . K(i)^T over this CTA's 256 latent (Q from TMEM) + 32 RoPE
    // columns, into S buffer i&1 once the softmax has read S(i-2) from it.
    // The scores run ahead of the softmax on their own; P.V comes from another
    // warp (MMA issue is nearly synchronous, so a wait in one issuer leaves
    // the tensor pipe to the other).
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      const uint64_t dqr = sdesc_sw64(sQR, 512);
      const uint64_t dk = sdesc_sw128(sKV, 16, 1024);
      const uint64_t dkr = sdesc_sw64(sKV + 4 * KV_CHUNK, 512);
      const uint32_t id_s = idesc_bf16(BM, BN, 0, 0);
      wait_or_fail(ok, bar(B_QFULL), 0, 11);
      wait_or_fail(ok, bar(B_QTMEM), 0, 15);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int s = i % STAGES, sb = i & (SBUF - 1);
        wait_or_fail(ok, bar(B_KVFULL + s), (i / STAGES) & 1, 12);
        if (i >= SBUF) wait_or_fail(ok, bar(B_SFREE + sb), ((i - SBUF) / SBUF) & 1, 13);
        if (!ok) break;
        // gathered tiles were written by cp.async (generic proxy): order them
        // before the tensor core's reads
        if (SPARSE) fence_async_shared();
        tc_fence_after();
        const uint64_t soff = (uint64_t)(s * (KV_STAGE >> 4));
        const uint32_t d = tmem + TM_S + sb * BN;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          mma_bf16_tmem_a(d, tmem + TM_QL + 8 * kk,
                          dk + soff + (((kk >> 2) * KV_CHUNK + (kk & 3) * 32) >> 4), id_s, kk != 0);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) mma_bf16(d, dqr + 2 * ks, dkr + soff + 2 * ks, id_s, 1);
        mma_commit(bar(B_SFULL + sb));
      }
      // every MMA issued here has finished before tensor memory is released
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0);
    }
    cluster_wait();
    cluster_arrive();
  } else if (warp == 2) {
    // --------------------------------------------------------- P.V issuer
    // O += P(j) . V(j) over this CTA's 256 latent columns of the KV tile; the
    // stage is free afterwards (S(j) finished before the softmax made P(j)).
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      const uint64_t dv = sdesc_sw128(sKV, KV_CHUNK, 1024);
      const uint64_t dp = sdesc_sw128(sP, 16, 1024);
      const uint32_t id_o = idesc_bf16(BM, 256, 0, 1);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int sj = j % STAGES, pb = j & 1;
        wait_or_fail(ok, bar(B_PFULL + pb), (j >> 1) & 1, 14);
        if (!ok) break;
        if (SPARSE) fence_async_shared();
        tc_fence_after();
        const uint64_t soff = (uint64_t)(sj * (KV_STAGE >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_O, dp + 2 * ks, dv + soff + ks * 128, id_o, (j > 0 || ks > 0));
        mma_commit(bar(B_ODONE + pb));
        mma_commit(bar(B_KVEMPTY + sj));
      }
      mma_commit(bar(B_DRAIN + 1));
      mbar_wait(bar(B_DRAIN + 1), 0);
    }
    cluster_wait();
    cluster_arrive();
  } else if (warp >= XCHG_WARP0) {
    // ------------------------------------------------------- score exchange
    // One warp per TMEM lane quarter ships this CTA's partial scores of each
    // tile to the peer as soon as the score MMAs finish, up to two tiles ahead
    // of the softmax, so the softmax's own steps never wait on a copy.
    cluster_wait();  // the peer's exchange barriers are set up
    if (ntiles > 0) {
      bool ok = true;
      const int quarter = warp & 3;
      const int q = quarter * 32 + lane;
      const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
      const uint32_t block = (uint32_t)(quarter * XQUARTER);
      const uint32_t peer_x = mapa(sX, peer);
      const uint32_t peer_xfull = mapa(bar(B_XFULL), peer);
      for (int j = 0; j < ntiles; ++j) {
        const int sb = j & (SBUF - 1);
        wait_or_fail(ok, bar(B_SFULL + sb), (j / SBUF) & 1, 26);
        tc_fence_after();
        uint32_t h[BN / 2];  // the row's partials, rounded, as fp16 pairs
#pragma unroll
        for (int g = 0; g < BN / 32; ++g) {
          uint32_t v[32];
          tmem_ld16(tmem + lane_base + TM_S + sb * BN + 32 * g, *(uint32_t(*)[16])(v));
          tmem_ld16(tmem + lane_base + TM_S + sb * BN + 32 * g + 16, *(uint32_t(*)[16])(v + 16));
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __half2 x = round_partial(v[2 * e], v[2 * e + 1], p.sl2);
            h[16 * g + e] = *reinterpret_cast<const uint32_t*>(&x);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SFREE + sb));
        if (lane == 0) {
          bulk_wait_read();  // this warp's previous copy has left the staging block
          // the peer has read tile j-2 out of exchange buffer j&1
          if (j >= 2) wait_cluster_or_fail(ok, bar(B_XFREE + (j & 1)), ((j - 2) >> 1) & 1, 21);
        }
        __syncwarp();
#pragma unroll
        for (int g = 0; g < NWG; ++g)
#pragma unroll
          for (int k = 0; k < XCH; ++k) {
            const uint32_t* w = h + g * (CPT / 2) + 4 * k;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             sStg + xchg_offset(g, q, k)),
                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                         : "memory");
          }
        fence_async_shared();
        __syncwarp();
        if (lane == 0 && ok)
          bulk_copy_to_peer(peer_x + (j & 1) * X_BYTES + block, sStg + block, XQUARTER,
                            peer_xfull + 8 * (j & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (lane == 0) bulk_wait_read();
    }
    // every copy this warp sent has been read out of its staging block; the
    // peer waits for their landing itself
    __syncwarp();
    cluster_arrive();
  } else {
    // ------------------------------------------------- softmax warpgroups
    // NWG warpgroups: thread (wg, q) owns row q, score columns CPT*wg.. and O
    // (and latent Q) columns OPT*wg.. of this CTA's share.  Tile i's scores
    // are this CTA's partial (read again from TMEM, rounded as it was sent)
    // plus the peer's, which the exchange warps have usually delivered by then.
    const int wg = (warp - 3) >> 2;
    const int q = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const int c0 = CPT * wg;
    const int sm_tid = threadIdx.x - 96;
    const int row = row0 + q;
    const int l = min(row, p.R - 1) / p.H;
    const int last_t = T - p.L + l;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t peer_xfree = mapa(bar(B_XFREE), peer);
    bool ok = true;
    int armed = min(ntiles, 2), received = 0;  // exchange phases armed / completed
    float m_run = -INFINITY, l_part = 0.f;
    float s[CPT];
    // index-list mode: this warp's lane holds list entry c0 + lane of a tile
    const int32_t* list = SPARSE ? p.topk + ((size_t)b * p.L + l) * p.topk_k : nullptr;
    auto list_entry = [&](int i) {
      const int j = kv0 + i * BN + c0 + lane;
      return j < kv1 ? list[j] : -1;
    };
    int pos_next = -1;
    if (ntiles > 0) {
      // this CTA's latent query columns into TMEM as bf16 pairs (the fold wrote them)
      pdl_wait();
      // chunk k of this thread's 128 columns: 16 B of row q (rows past R hold
      // whatever the workspace held; they only feed their own, unused, rows)
      const uint4* src = (const uint4*)(p.q_lat) +
                         (((size_t)b * p.rtiles + tile) * 64 + 32 * rank + (OPT / 8) * wg) * 128 +
                         q;
#pragma unroll
      for (int k = 0; k < OPT / 64; ++k) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = src[(size_t)(8 * k + u) * 128];
          v[4 * u] = x.x;
          v[4 * u + 1] = x.y;
          v[4 * u + 2] = x.z;
          v[4 * u + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + TM_QL + (OPT / 2) * wg + 32 * k, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_QTMEM));
      if (SPARSE) pos_next = list_entry(0);
      load_partial(ok, tmem, lane_base, c0, 0, bar(B_SFULL), bar(B_SFREE), p.sl2, s);
    }
    cluster_wait();  // the peer's barriers are set up before the first remote arrive
    // One tile of the softmax; `s` holds tile i's own (rounded) partial on
    // entry and tile i+1's on exit (read once P(i) is out, so only one tile's
    // scores are ever live in registers).
    for (int i = 0; i < ntiles; ++i) {
      const int t0 = kv0 + i * BN;
      // finish tile i's scores with the peer's partial; the causal verify mask
      // only matters on tiles that reach past the first row's last position
      const bool edge = t0 + BN - 1 > T - p.L;
      const int xb = i & 1;  // exchange buffer of tile i
      wait_cluster_or_fail(ok, bar(B_XFULL + xb), (i >> 1) & 1, 22);
      if (ok) received = i + 1;
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < XCH; ++k) {
        uint32_t h[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
                     : "r"(sX + xb * X_BYTES + xchg_offset(wg, q, k)));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
          const int j = 8 * k + 2 * e;
          s[j] += f.x;
          s[j + 1] += f.y;
        }
      }
      if (SPARSE) {
        // every row of the tile is one verify row: one mask per warp
        const uint32_t vm = __ballot_sync(0xffffffffu, pos_next >= 0 && pos_next <= last_t);
        if (i + 1 < ntiles) pos_next = list_entry(i + 1);
#pragma unroll
        for (int j = 0; j < CPT; ++j) s[j] = ((vm >> j) & 1u) ? s[j] : -INFINITY;
      } else if (edge) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) s[j] = (t0 + c0 + j <= last_t) ? s[j] : -INFINITY;
      }
      float m2[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int j = 4; j < CPT; ++j) m2[j & 3] = fmaxf(m2[j & 3], s[j]);
      mt = fmaxf(fmaxf(m2[0], m2[1]), fmaxf(m2[2], m2[3]));
      red[wg * BM + q] = mt;
      named_bar_sync(1, SOFTMAX_THREADS);  // exchange tile read by all; row maxima visible
#pragma unroll
      for (int g = 0; g < NWG; ++g) mt = fmaxf(mt, red[g * BM + q]);
      if (sm_tid == 0 && ok) {
        if (i + 2 < ntiles) {
          mbar_arrive_expect_tx(bar(B_XFULL + xb), X_BYTES);  // arm buffer xb for tile i+2
          ++armed;
        }
        // the peer may now send tile i+2 into buffer xb: every read of it has
        // returned (its values were used before the bar.sync), so no fence
        mbar_arrive_remote_relaxed(peer_xfree + 8 * xb);
      }
    // lazy rescale: move the running max only when it grows by more than 2^8;
      // O must then hold every earlier P.V
      const bool need = mt > m_run + 8.f;
      const float m_new = need ? mt : m_run;
      const float factor = need ? ex2(m_run - m_new) : 1.f;
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        wait_or_fail(ok, bar(B_ODONE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, 23);
        tc_fence_after();
        for (int c = 0; c < OPT; c += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + TM_O + OPT * wg + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * factor);
          tmem_st16(tmem + lane_base + TM_O + OPT * wg + c, v);
        }
        tmem_wait_st();
      }
      l_part *= factor;
      m_run = m_new;
      // P = 2^(s - m) in bf16 into the P tile (K-major, 128-byte swizzled rows),
      // which P.V(i-1) has finished reading
      if (i >= 1) wait_or_fail(ok, bar(B_ODONE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, 24);
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float rs[2] = {0.f, 0.f};
      const uint32_t prow = sP + q * 128;
#pragma unroll
      for (int k = 0; k < CPT / 8; ++k) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = ex2(s[8 * k + 2 * e] - m_use);
          const float d = ex2(s[8 * k + 2 * e + 1] - m_use);
          rs[0] += a;
          rs[1] += d;
          pk[e] = pack_bf16(a, d);
        }
        const int c = (c0 >> 3) + k;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + (((c ^ q) & 7) << 4)),
                     "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                     : "memory");
      }
      l_part += rs[0] + rs[1];
      // positions at or past T in the last tile: zero their value rows (they may hold
      // anything, and 0 * NaN would poison the accumulator)
      if (!SPARSE && t0 + BN > T) {
        const int z0 = max(T - t0, 0);
        const uint32_t st = sKV + (i % STAGES) * KV_STAGE;
        const int units = (BN - z0) * 8;  // 16-byte units per 128-byte row
        for (int u = sm_tid; u < 4 * units; u += SOFTMAX_THREADS) {
          const int c = u / units, w = u - c * units;
          const uint32_t addr = st + c * KV_CHUNK + (z0 + w / 8) * 128 + (w & 7) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                       : "memory");
        }
      }
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + (i & 1)));
      // this CTA's partial of tile i+1
      if (i + 1 < ntiles)
        load_partial(ok, tmem, lane_base, c0, i + 1, bar(B_SFULL), bar(B_SFREE), p.sl2, s);
    }
    // after a failure, let an armed exchange phase finish (or time out) so no
    // copy from the peer is still landing when this CTA exits
    if (sm_tid == 0)
      for (int j = received; j < armed; ++j)
        mbar_wait_cluster(bar(B_XFULL + (j & 1)), (j >> 1) & 1);
    // the last remote arrive of this warpgroup is done: the exit barrier's
    // arrival (the epilogue below touches only this CTA)
    __syncwarp();
    cluster_arrive();
    // ---------------------------------------------------------------- epilogue
    if (ntiles > 0) wait_or_fail(ok, bar(B_ODONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, 25);
    pdl_wait();  // the partials may still be read by the previous call's merge
    tc_fence_after();
    const bool live = row < p.R;
    // The row's total l: the sum of the two warpgroups' shares (both CTAs of the
    // pair hold the same P, so their totals agree).
    lsum[wg * BM + q] = l_part;
    named_bar_sync(1, SOFTMAX_THREADS);
    float l_tot = 0.f;
#pragma unroll
    for (int g = 0; g < NWG; ++g) l_tot += lsum[g * BM + q];
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    // This CTA's half of O / l (128 rows x 256 columns, bf16) goes through the
    // drained KV stages as four 128-byte-swizzled boxes of 64 columns, then
    // out with TMA stores (rows past R are clipped).
    // (64 columns per round: four TMEM loads in flight, one wait)
    for (int c = 0; c < OPT; c += 64) {
      uint32_t v[64];
      if (ntiles > 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tmem_ld16(tmem + lane_base + TM_O + OPT * wg + c + 16 * k,
                    *(uint32_t(*)[16])(v + 16 * k));
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] = 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int col = OPT * wg + c + 8 * u;
        const uint32_t addr = sKV + (col >> 6) * (BM * 128) + q * 128 +
                              ((((col & 63) >> 3) ^ (q & 7)) << 4);
        const uint32_t* w = v + 8 * u;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                     "r"(pack_bf16(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv)),
                     "r"(pack_bf16(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv)),
                     "r"(pack_bf16(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv)),
                     "r"(pack_bf16(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv))
                     : "memory");
      }
    }
    fence_async_shared();
    named_bar_sync(1, SOFTMAX_THREADS);
    if (sm_tid == 0) {
      for (int bx = 0; bx < 4; ++bx)
        tma_store_3d(&tm_op, sKV + bx * (BM * 128), (int)rank * 256 + 64 * bx, row0,
                     b * p.splits + split);
      bulk_commit();
      // the staging may be released once the stores have read it; their
      // writes are complete when the grid is (the merge reads them after its
      // dependency wait)
      bulk_wait_read();
    }
    if (live && rank == 0 && wg == 0) {
      float* mlp = p.ml + (((size_t)b * p.splits + split) * p.R + row) * 2;
      mlp[0] = m_run == -INFINITY ? -FLT_MAX : m_run;
      mlp[1] = l_tot;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // no peer access may outlive this CTA: every thread of both CTAs arrived
  // once its accesses to the peer were done
  cluster_wait();
}

// =========================================================================
// merge of the split-KV pieces
// =========================================================================
// o_lat[row] = sum_s w_s (O_s / l_s)[row] / sum_s w_s with w_s = 2^(m_s - M) l_s
// (bf16 out).  One CTA per (query row, 256*CPL-column slice): warp w takes every
// W-th piece, each lane CPL groups of 8 columns, with its own running maximum
// (raised, and the sums rescaled, when a piece's maximum is larger), so there
// is no separate max pass and the loads of many pieces are in flight at once;
// the W warps' sums are combined in shared memory.  The launcher uses CPL = 1
// (two CTAs per row: more CTAs, fewer loads each) with eight warps for rows of
// 48 pieces or more and four for 32 to 47, CPL = 2 (one CTA per row) for 16 to
// 31, and sends rows with fewer to merge_rows_sm103 below, one warp per row.
struct MergeParams {
  const __nv_bfloat16* o_part;  // [B, splits, R, 512]
  const float* ml;              // [B, splits, R, 2]
  const int32_t* lens;
  __nv_bfloat16* o_lat;         // [B*R, 512]
  int R, chunk, splits;
  int rows;                     // B*R
  int fixed_len;                // > 0: every sequence's pieces split this many list entries
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int CPL, int W>  // W warps take every W-th piece
__global__ void __launch_bounds__(32 * W) merge_sm103(MergeParams p) {
  constexpr int NBATCH = 64 / (CPL * W);  // pieces whose loads are in flight together
  __shared__ float part[W][CPL * 8][32];
  __shared__ float mden[W][2];
  // the unembedding may start loading its weights now; it waits for this grid
  // before reading o_lat
  pdl_launch_dependents();
  const int rg = blockIdx.x;  // b*R + row
  const int col0 = blockIdx.y * 256 * CPL;
  const int b = rg / p.R, row = rg - b * p.R;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the length is a call input: read it while the attention finishes, so the
  // pieces' loads are the only round trip after the wait
  const int nsplit = ((p.fixed_len > 0 ? p.fixed_len : p.lens[b]) + p.chunk - 1) / p.chunk;
  pdl_wait();
  const size_t base = (size_t)b * p.splits * p.R + row;
  const size_t stride = (size_t)p.R;
  float M = -FLT_MAX, den = 0.f;
  float acc[CPL][8];
#pragma unroll
  for (int c = 0; c < CPL; ++c)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
  for (int s0 = w; s0 < nsplit; s0 += W * NBATCH) {
    float2 mls[NBATCH];
    uint4 x[NBATCH][CPL];
#pragma unroll
    for (int k = 0; k < NBATCH; ++k) {
      const int s = s0 + W * k;
      const size_t e = base + (size_t)min(s, nsplit - 1) * stride;
      mls[k] = *(const float2*)(p.ml + e * 2);
      const __nv_bfloat16* o = p.o_part + e * kLat + col0 + 8 * lane;
#pragma unroll
      for (int c = 0; c < CPL; ++c) x[k][c] = *(const uint4*)(o + 256 * c);
      if (s >= nsplit) mls[k].y = 0.f;  // past the last piece: weight 0
    }
#pragma unroll
    for (int k = 0; k < NBATCH; ++k) {
      if (mls[k].y > 0.f) {
        if (mls[k].x > M) {  // warp-uniform: every lane reads the same (m, l)
          const float f = ex2(M - mls[k].x);
          M = mls[k].x;
          den *= f;
#pragma unroll
          for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[c][e] *= f;
        }
        const float wt = ex2(mls[k].x - M) * mls[k].y;
        den += wt;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float f[8];
          bf16x8_to_f32(x[k][c], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[c][e] += wt * f[e];
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c)
#pragma unroll
    for (int e = 0; e < 8; ++e) part[w][8 * c + e][lane] = acc[c][e];
  if (lane == 0) {
    mden[w][0] = M;
    mden[w][1] = den;
  }
  __syncthreads();
  if (w == 0) {
    float Mall = mden[0][0];
#pragma unroll
    for (int g = 1; g < W; ++g) Mall = fmaxf(Mall, mden[g][0]);
    float f[W], dsum = 0.f;
#pragma unroll
    for (int g = 0; g < W; ++g) {
      f[g] = mden[g][1] > 0.f ? ex2(mden[g][0] - Mall) : 0.f;
      dsum += f[g] * mden[g][1];
    }
    const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float a = 0.f;
#pragma unroll
        for (int g = 0; g < W; ++g) a += f[g] * part[g][8 * c + e][lane];
        y[e] = a * inv;
      }
      *(uint4*)(p.o_lat + (size_t)rg * kLat + col0 + 256 * c + 8 * lane) =
          make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                     pack_bf16(y[6], y[7]));
    }
  }
}

// Few pieces per row: one warp per row over all its pieces (lane c owns
// columns 8c..8c+7 and 256+8c..256+8c+7), eight pieces' loads in flight per
// lane, so no shared memory and no barrier; four rows per CTA.
constexpr int MR_ROWS = 4;
__global__ void __launch_bounds__(32 * MR_ROWS) merge_rows_sm103(MergeParams p) {
  pdl_launch_dependents();  // the unembedding may start loading its weights
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = blockIdx.x * MR_ROWS + w;  // b*R + row
  const bool live = rg < p.rows;
  const int b = live ? rg / p.R : 0, row = rg - b * p.R;
  // (the length is a call input: read it before the wait)
  const int nsplit =
      live ? ((p.fixed_len > 0 ? p.fixed_len : p.lens[b]) + p.chunk - 1) / p.chunk : 0;
  pdl_wait();
  if (!live) return;
  const size_t base = (size_t)b * p.splits * p.R + row;
  float M = -FLT_MAX, den = 0.f, acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float2 mls[8];
    uint4 x[8][2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const size_t e = base + (size_t)min(s0 + j, nsplit - 1) * p.R;
      mls[j] = *(const float2*)(p.ml + e * 2);
      const __nv_bfloat16* o = p.o_part + e * kLat + 8 * lane;
      x[j][0] = *(const uint4*)(o);
      x[j][1] = *(const uint4*)(o + 256);
      if (s0 + j >= nsplit) mls[j].y = 0.f;  // past the last piece: weight 0
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (mls[j].y > 0.f) {
        if (mls[j].x > M) {  // warp-uniform: every lane reads the same (m, l)
          const float f = ex2(M - mls[j].x);
          M = mls[j].x;
          den *= f;
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] *= f;
        }
        const float wt = ex2(mls[j].x - M) * mls[j].y;
        den += wt;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float f[8];
          bf16x8_to_f32(x[j][half], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[8 * half + e] += wt * f[e];
        }
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float* a = acc + 8 * half;
    *(uint4*)(p.o_lat + (size_t)rg * kLat + 256 * half + 8 * lane) =
        make_uint4(pack_bf16(a[0] * inv, a[1] * inv), pack_bf16(a[2] * inv, a[3] * inv),
                   pack_bf16(a[4] * inv, a[5] * inv), pack_bf16(a[6] * inv, a[7] * inv));
  }
}

// =========================================================================
// unembedding + merge of the split-KV pieces
// =========================================================================
// The merge and the unembedding commute.  With the combine weights of row
// (l, h) of sequence b over its pieces s,
//   w_{l,s} = 2^(m_s - M_l) l_s / sum_s' 2^(m_s' - M_l) l_s',
//   out[b, l, h, :] = (sum_s w_{l,s} (O_s / l_s)[l, h, :]) . W_UV[h]
//                   = sum_s w_{l,s} ((O_s / l_s)[l, h, :] . W_UV[h]).
// One CTA per (head h, 128-column tile mt, block of sequences).  Its W_UV
// tile (K = 512 rows, MN-major) is loaded with TMA before the dependency
// wait (W_UV does not depend on the attention, which also pulled it into
// L2).  After the wait, chunk after chunk: one 4-D TMA box brings the bf16
// rows (O_s / l_s)[l, h, :] of every piece s of Lc verify rows of one
// sequence (rows ordered by l, then s; Lc * splits <= 64) into shared memory
// as the K-major B operand, and one GEMM D[128 x rows] = W_UV tile^T x rows^T
// lands in one of two 64-column TMEM slabs.  Meanwhile three warps compute
// every chunk's combine weights from (m, l), in the chunk's column order; the
// epilogue warpgroup sums each verify row's columns with them and writes the
// row.  All the piece rows of a chunk are in flight at once, and o_lat is
// never formed.
struct UnembedMergeParams {
  const float* ml;        // [B, splits, R, 2]
  const int32_t* lens;
  __nv_bfloat16* out;     // [B, L, H, v]
  int B, L, H, R, v, splits, chunk;
  int Lc;                 // verify rows per chunk (Lc * splits <= 64)
  int chunks_per_cta;     // consecutive chunks of the (sequence, verify-row block) list
  int fixed_len;          // > 0: every sequence's pieces split this many list entries
};
constexpr int UM_THREADS = 256;            // warp 0 issues, 1..3 weights, 4..7 epilogue
constexpr int UM_W = 2 * kLat * 128;       // W_UV tile
constexpr int UM_B = 8 * 64 * 128;         // one chunk of at most 64 piece rows
constexpr int UM_MAX_CHUNKS = 64;          // chunks per CTA (weights table of 16 KB)
constexpr int UM_OFF_B = UM_W;
constexpr int UM_OFF_WT = UM_OFF_B + UM_B;
constexpr int UM_OFF_BAR = UM_OFF_WT + UM_MAX_CHUNKS * 64 * 4;
constexpr int UM_SMEM = UM_OFF_BAR + 128 + 1024;
static_assert(UM_SMEM <= 232448, "shared memory per CTA");
enum { UB_WFULL = 0, UB_OFULL = 1, UB_DONE = 2, UB_FREE = 4, UB_COUNT = 6 };

// Combine weights of every (chunk, verify row) of a CTA, one thread of warps
// 1..3 per row, for rows of up to 32 pieces.
__device__ __forceinline__ void um_weights_many_rows(const UnembedMergeParams& p, float* wts, int h,
                                                  int g0, int nch, int cps, int Lc, int S) {
  for (int row = threadIdx.x - 32; row < nch * Lc; row += 96) {
    const int c = row / Lc, li = row - c * Lc;
    const int b = (g0 + c) / cps, l = ((g0 + c) % cps) * Lc + li;
    float* wt = wts + c * 64 + li * S;
    const int len = p.fixed_len > 0 ? p.fixed_len : p.lens[b];
    const int nsplit = l < p.L ? min((len + p.chunk - 1) / p.chunk, S) : 0;
    const float2* mlr = (const float2*)p.ml + (size_t)b * S * p.R +
                        (size_t)min(l, p.L - 1) * p.H + h;
    float M = -FLT_MAX;
    for (int j0 = 0; j0 < nsplit; j0 += 8) {
      float2 e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        e[j] = j0 + j < nsplit ? mlr[(size_t)(j0 + j) * p.R] : make_float2(-FLT_MAX, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e[j].y > 0.f) M = fmaxf(M, e[j].x);
    }
    float sum = 0.f;
    for (int j0 = 0; j0 < S; j0 += 8) {
      float2 e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        e[j] = j0 + j < nsplit ? mlr[(size_t)(j0 + j) * p.R] : make_float2(-FLT_MAX, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = e[j].y > 0.f ? ex2(e[j].x - M) * e[j].y : 0.f;
        sum += w;
        if (j0 + j < S) wt[j0 + j] = w;
      }
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int j = 0; j < S; ++j) wt[j] *= inv;
  }
}

// MANY_ROWS: the instantiation for CTAs with many rows of 9 to 32 pieces
// (batches of long caches), which computes their weights one thread per row;
// the other instantiation, without that code, serves everything else.
template <bool MANY_ROWS>
__global__ void __launch_bounds__(UM_THREADS, 1)
    unembed_merge_sm103(const __grid_constant__ CUtensorMap tm_wuv,
                        const __grid_constant__ CUtensorMap tm_pieces, UnembedMergeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sW = smem_u32(smem), sB = smem_u32(smem + UM_OFF_B);
  float* wts = (float*)(smem + UM_OFF_WT);  // [chunk][64] weights in column order
  uint64_t* bars = (uint64_t*)(smem + UM_OFF_BAR);
  uint32_t* slot = (uint32_t*)(bars + UB_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nmt = p.v / 128;
  const int h = blockIdx.x / nmt, mt = blockIdx.x - h * nmt;
  const int S = p.splits, Lc = p.Lc;
  const int cps = (p.L + Lc - 1) / Lc;  // chunks per sequence
  // this CTA's chunks: g0 .. g0 + nch - 1 of the B * cps chunks, sequence by
  // sequence; chunk g is verify rows (g % cps) * Lc .. of sequence g / cps
  const int g0 = blockIdx.y * p.chunks_per_cta;
  const int nch = min(p.chunks_per_cta, p.B * cps - g0);

  if (threadIdx.x == 0) {
    mbar_init(bar(UB_WFULL), 1);
    mbar_init(bar(UB_OFULL), 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(UB_DONE + k), 1);
      mbar_init(bar(UB_FREE + k), 128);
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  pdl_launch_dependents();  // the next kernel may start its own independent loads

  if (warp == 0) {
    // ------------------------------------------------ TMA + MMA issue (one thread)
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(bar(UB_WFULL), UM_W);
      for (int kc = 0; kc < kLat / 64; ++kc)
        for (int j = 0; j < 2; ++j)
          tma_load_2d(sW + j * kLat * 128 + kc * 8192, &tm_wuv, bar(UB_WFULL), mt * 128 + 64 * j,
                      h * kLat + 64 * kc);
      pdl_wait();  // the pieces come from the attention
      const uint32_t slab = 128u * S * Lc;
      const int N = (S * Lc + 15) & ~15;
      const uint32_t idesc = idesc_bf16(128, N, 1, 0);
      for (int c = 0; c < nch && ok; ++c) {
        const int b = (g0 + c) / cps, l0 = ((g0 + c) % cps) * Lc;
        mbar_arrive_expect_tx(bar(UB_OFULL), 8 * slab);
        for (int kc = 0; kc < kLat / 64; ++kc)
          tma_load_4d(sB + kc * 8192, &tm_pieces, bar(UB_OFULL), 64 * kc, h, b * S, l0);
        wait_or_fail(ok, bar(UB_OFULL), c & 1, 50);
        if (c == 0) wait_or_fail(ok, bar(UB_WFULL), 0, 51);
        if (c >= 2) wait_or_fail(ok, bar(UB_FREE + (c & 1)), ((c - 2) >> 1) & 1, 52);
        if (!ok) break;
        tc_fence_after();
        for (int kc = 0; kc < kLat / 64; ++kc)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + 64 * (c & 1),
                     sdesc_sw128(sW + (kc * 64 + ks * 16) * 128, kLat * 128, 1024),
                     sdesc_sw128(sB + kc * 8192 + ks * 32, 16, 1024), idesc, (kc | ks) != 0);
        mma_commit(bar(UB_DONE + (c & 1)));
        // the chunk buffer is free for the next box once these MMAs are done
        wait_or_fail(ok, bar(UB_DONE + (c & 1)), (c >> 1) & 1, 53);
        if (!ok) break;
      }
      // nothing this thread started may still be landing when the CTA exits
      mbar_wait(bar(UB_WFULL), 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------ combine weights (3 warps)
    pdl_wait();
    if (S <= 8) {
      // few pieces per row (wide verify widths): one thread per row, its
      // pieces' (m, l) loads all in flight at once
      for (int row = threadIdx.x - 32; row < nch * Lc; row += 96) {
        const int c = row / Lc, li = row - c * Lc;
        const int b = (g0 + c) / cps, l = ((g0 + c) % cps) * Lc + li;
        float* wt = wts + c * 64 + li * S;
        const int len = p.fixed_len > 0 ? p.fixed_len : p.lens[b];
        const int nsplit = l < p.L ? (len + p.chunk - 1) / p.chunk : 0;
        const size_t base = (size_t)b * S * p.R + (size_t)min(l, p.L - 1) * p.H + h;
        float2 ml[8];
        float M = -FLT_MAX;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          ml[j] = j < nsplit && j < S ? *(const float2*)(p.ml + (base + (size_t)j * p.R) * 2)
                                      : make_float2(-FLT_MAX, 0.f);
          if (ml[j].y > 0.f) M = fmaxf(M, ml[j].x);
        }
        float w[8], sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          w[j] = ml[j].y > 0.f ? ex2(ml[j].x - M) * ml[j].y : 0.f;
          sum += w[j];
        }
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < S) wt[j] = w[j] * inv;
      }
    } else if (MANY_ROWS && S <= 32) {
      // many rows of up to 32 pieces (two passes of S/8 round trips to memory
      // per row beat the warp-per-row form's rows/3 round trips):
      // one thread per row, eight pieces' (m, l) loads in flight per batch:
      // the row maximum first, then the weights (the second read hits L1),
      // normalised in shared memory.  (The warp-per-row form below walked a
      // CTA's rows three at a time, one round trip to memory each: 237 us
      // against 173 for the batched serving call's unembedding.)
      um_weights_many_rows(p, wts, h, g0, nch, cps, Lc, S);
    } else {
      for (int row = warp - 1; row < nch * Lc; row += 3) {  // (chunk, verify row in it)
        const int c = row / Lc, li = row - c * Lc;
        const int b = (g0 + c) / cps, l = ((g0 + c) % cps) * Lc + li;
        float* wt = wts + c * 64 + li * S;
        if (l >= p.L) {
          for (int s = lane; s < S; s += 32) wt[s] = 0.f;
          continue;
        }
        const int nsplit = ((p.fixed_len > 0 ? p.fixed_len : p.lens[b]) + p.chunk - 1) / p.chunk;
        const size_t base = (size_t)b * S * p.R + (size_t)l * p.H + h;
        float2 ml[2];
        float M = -FLT_MAX;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int sj = lane + 32 * j;
          ml[j] = sj < nsplit ? *(const float2*)(p.ml + (base + (size_t)sj * p.R) * 2)
                              : make_float2(-FLT_MAX, 0.f);
          if (ml[j].y > 0.f) M = fmaxf(M, ml[j].x);
        }
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, o));
        float w[2], sum = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          w[j] = ml[j].y > 0.f ? ex2(ml[j].x - M) * ml[j].y : 0.f;
          sum += w[j];
        }
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(~0u, sum, o);
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
          if (lane + 32 * j < S) wt[lane + 32 * j] = w[j] * inv;
      }
    }
    named_bar_sync(1, 224);  // weights -> epilogue
  } else {
    // ------------------------------------------------ epilogue (one warpgroup)
    // TMEM lane m is output column 128 mt + m; a chunk's column j is piece
    // j % S of its verify row j / S.  Pieces past a sequence's last have
    // weight 0 and rows that were never written: they are skipped, not
    // multiplied (the rows may hold anything).
    named_bar_sync(1, 224);
    const int m = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      const int b = (g0 + c) / cps, l0 = ((g0 + c) % cps) * Lc;
      const int rows = min(Lc, p.L - l0) * S;
      wait_or_fail(ok, bar(UB_DONE + (c & 1)), (c >> 1) & 1, 54);
      tc_fence_after();
      if (ok) {
        __nv_bfloat16* o = p.out + (((size_t)b * p.L + l0) * p.H + h) * p.v + mt * 128 + m;
        const float* wt = wts + c * 64;
        float acc = 0.f;
        int row_end = S - 1, l = 0;
        for (int j0 = 0; j0 < rows; j0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + 64 * (c & 1) + j0, v);
          float wv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 w4 = *(const float4*)(wt + j0 + 4 * q);
            wv[4 * q] = w4.x;
            wv[4 * q + 1] = w4.y;
            wv[4 * q + 2] = w4.z;
            wv[4 * q + 3] = w4.w;
          }
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = j0 + e;
            if (j < rows) {
              if (wv[e] != 0.f) acc = fmaf(wv[e], __uint_as_float(v[e]), acc);
              if (j == row_end) {  // verify row l0 + l complete
                o[(size_t)l * p.H * p.v] = __float2bfloat16_rn(acc);
                acc = 0.f;
                row_end += S;
                ++l;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(UB_FREE + (c & 1)));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// Per-device one-time setup: the kernels' shared-memory opt-in and the number
// of attention clusters that fit on the device at once (the piece planner
// sizes its grid with it).  Calls may come from several threads; the first
// one on a device does the work under a lock.
struct DeviceSetup {
  cudaError_t err = cudaSuccess;
  int slots = 0;
  bool done = false;
};

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

bool fast_absorbed_supported(const Plan& p) {
  return p.dtype == MLA_DTYPE_BF16 && p.r == kLat && p.rope == 64 && p.n % 64 == 0 &&
         p.n >= 64 && p.n <= 256 && p.v % 128 == 0 && p.v <= 512;
}

namespace {

// Rows per CTA of the swap-AB GEMM: the whole batch up to 256 (64 when K is
// 512, so the weight tile and the activations fit in shared memory).
int gemm_rows(int BL, int K) {
  const int cap = K >= 512 ? 64 : 256;
  const int nb = ((BL + 15) / 16) * 16;
  return nb > cap ? cap : nb;
}

int gemm_smem(int K, int NB) { return 2 * K * 128 + (K / 64) * NB * 128 + 1024 + 128; }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

const DeviceSetup& device_setup() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static DeviceSetup setups[kMaxDevices];
  static DeviceSetup no_device;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    no_device.slots = device_sm_count() / 2;
    no_device.err = cudaErrorNoDevice;
    return no_device;
  }
  std::lock_guard<std::mutex> lk(mu);
  DeviceSetup& d = setups[dev];
  if (d.done) return d;
  cudaError_t e = set_smem(swapab_gemm_sm103, gemm_smem(kLat, 64));
  if (e == cudaSuccess) e = set_smem(absorbed_attn_sm103<false>, ATTN_SMEM);
  if (e == cudaSuccess) e = set_smem(absorbed_attn_sm103<true>, ATTN_SMEM);
  if (e == cudaSuccess) e = set_smem(unembed_merge_sm103<false>, UM_SMEM);
  if (e == cudaSuccess) e = set_smem(unembed_merge_sm103<true>, UM_SMEM);
  int slots = 0;
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(ATTN_THREADS);
    cfg.dynamicSmemBytes = ATTN_SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&slots, absorbed_attn_sm103<false>, &cfg) != cudaSuccess)
      slots = 0;
  }
  if (slots <= 0) {
    cudaGetLastError();
    slots = device_sm_count() / 2;
  }
  d.err = e;
  d.slots = slots;
  d.done = true;
  return d;
}

}  // namespace

int absorbed_cluster_slots() { return device_setup().slots; }

cudaError_t launch_fast_absorbed(const Plan& p, const Args& a) {
  const int BL = p.B * p.L;
  const int R = p.L * p.H;
  __nv_bfloat16* q_lat = (__nv_bfloat16*)(a.ws + p.off_qlat);
  __nv_bfloat16* o_part = (__nv_bfloat16*)(a.ws + p.off_opart);
  float* ml = (float*)(a.ws + p.off_ml);
  __nv_bfloat16* o_lat = (__nv_bfloat16*)(a.ws + p.off_olat);
  const CacheView& c = a.cache;
  const long long cache_rows =
      c.page_table ? (long long)c.num_pages * c.page_size
                   : (long long)(p.B - 1) * c.seq_stride + p.Tmax;

  CUtensorMap tm_wuk, tm_qn, tm_qr, tm_ckv, tm_kr, tm_wuv, tm_ol, tm_op;
  const int NBf = gemm_rows(BL, p.n), NBu = gemm_rows(BL, kLat);
  bool ok = make_tmap_bf16_2d(&tm_wuk, a.W_UK, kLat, (uint64_t)p.H * p.n, kLat * 2, 64, 64, 128);
  ok = ok && make_tmap_bf16_2d(&tm_qn, a.q_nope, (uint64_t)p.H * p.n, BL, (uint64_t)p.H * p.n * 2,
                               64, NBf, 128);
  ok = ok && make_tmap_bf16_2d(&tm_qr, a.q_rope, 64, (uint64_t)p.B * R, 128, 32, BM, 64);
  ok = ok && make_tmap_bf16_2d(&tm_ckv, c.c_kv, kLat, cache_rows, c.ckv_stride * 2, 64, BN, 128);
  ok = ok && make_tmap_bf16_2d(&tm_kr, c.k_rope, 64, cache_rows, c.kr_stride * 2, 32, BN, 64);
  ok = ok && make_tmap_bf16_2d(&tm_wuv, a.W_UV, p.v, (uint64_t)p.H * kLat, (uint64_t)p.v * 2, 64,
                               64, 128);
  ok = ok && make_tmap_bf16_2d(&tm_ol, o_lat, (uint64_t)p.H * kLat, BL, (uint64_t)p.H * kLat * 2,
                               64, NBu, 128);
  ok = ok && make_tmap_bf16_3d(&tm_op, o_part, kLat, R, (uint64_t)p.B * p.splits, kLat * 2,
                               (uint64_t)R * kLat * 2, 64, BM);
  if (!ok) return cudaErrorInvalidValue;

  const DeviceSetup& ds = device_setup();
  if (ds.err != cudaSuccess) return ds.err;
  cudaError_t e;
  {
    GemmParams gp{q_lat, BL, p.H, p.n, kLat, NBf, p.L, (R + BM - 1) / BM};
    KernelTimer kt("fold_sm103", a.stream);
    e = launch_pdl(swapab_gemm_sm103, dim3(kLat / 128, p.H, (BL + NBf - 1) / NBf), dim3(128),
                   gemm_smem(p.n, NBf), a.stream, tm_wuk, tm_qn, gp);
    if (e != cudaSuccess) return e;
  }
  {
    AttnParams ap;
    ap.lens = a.lens;
    ap.page_table = c.page_table;
    ap.q_lat = q_lat;
    ap.B = p.B;
    ap.page_size = c.page_size;
    ap.max_pages = c.max_pages;
    ap.num_pages = c.num_pages;
    ap.seq_stride = c.seq_stride;
    ap.L = p.L;
    ap.H = p.H;
    ap.R = R;
    ap.rtiles = (R + BM - 1) / BM;
    ap.chunk = p.chunk;
    ap.splits = p.splits;
    ap.sl2 = p.scale * 1.4426950408889634f;
    ap.o_part = o_part;
    ap.ml = ml;
    ap.pf = (const char*)a.W_UV;
    ap.pf_bytes = (size_t)p.H * kLat * p.v * 2;
    ap.topk = a.topk;
    ap.topk_k = a.topk_k;
    ap.ckv = (const char*)c.c_kv;
    ap.kr = (const char*)c.k_rope;
    ap.ckv_stride = c.ckv_stride;
    ap.kr_stride = c.kr_stride;
    const dim3 grid(2 * ((R + BM - 1) / BM), p.splits, p.B);
    if (a.topk) {
      KernelTimer kt("absorbed_attn_sparse_sm103", a.stream);
      e = launch_pdl(absorbed_attn_sm103<true>, grid, dim3(ATTN_THREADS), ATTN_SMEM, a.stream,
                     tm_qr, tm_ckv, tm_kr, tm_op, ap);
    } else {
      KernelTimer kt("absorbed_attn_sm103", a.stream);
      e = launch_pdl(absorbed_attn_sm103<false>, grid, dim3(ATTN_THREADS), ATTN_SMEM, a.stream,
                     tm_qr, tm_ckv, tm_kr, tm_op, ap);
    }
    if (e != cudaSuccess) return e;
  }
  if (p.splits <= 64) {
    // unembedding + merge in one kernel
    UnembedMergeParams up;
    up.ml = ml;
    up.lens = a.lens;
    up.out = (__nv_bfloat16*)a.out;
    up.B = p.B;
    up.L = p.L;
    up.H = p.H;
    up.R = R;
    up.v = p.v;
    up.splits = p.splits;
    up.chunk = p.chunk;
    up.Lc = 64 / p.splits < p.L ? 64 / p.splits : p.L;
    // chunks per CTA: one wave of CTAs (each loads its 128 KB W_UV tile
    // once for all of its chunks), at most UM_MAX_CHUNKS
    const int units = p.H * (p.v / 128);
    const int cps = (p.L + up.Lc - 1) / up.Lc;
    const long long total = (long long)p.B * cps;
    const long long want_ctas = device_sm_count();  // one CTA fits an SM
    long long cpc = (total * units + want_ctas - 1) / want_ctas;
    if (cpc < 1) cpc = 1;
    if (cpc > UM_MAX_CHUNKS) cpc = UM_MAX_CHUNKS;
    up.chunks_per_cta = (int)cpc;
    up.fixed_len = a.topk ? a.topk_k : 0;
    {
      // the pieces of one head as [l][piece][h][col]: row (b, s, l, h) of
      // o_part sits at ((b * splits + s) * R + l * H + h) * 512 elements
      CUtensorMap tm_pieces;
      const uint64_t dims[4] = {(uint64_t)kLat, (uint64_t)p.H, (uint64_t)p.B * p.splits,
                                (uint64_t)p.L};
      const uint64_t strides[3] = {(uint64_t)kLat * 2, (uint64_t)R * kLat * 2,
                                   (uint64_t)p.H * kLat * 2};
      const uint32_t box[4] = {64, 1, (uint32_t)p.splits, (uint32_t)up.Lc};
      if (!make_tmap_bf16_4d(&tm_pieces, o_part, dims, strides, box)) return cudaErrorInvalidValue;
      // rows of 9 to 32 pieces, many per CTA: two passes of S/8 round trips to
      // memory per row (one thread each) beat one round trip per three rows
      const long long rows_per_cta = cpc * up.Lc;
      const bool many_rows = p.splits > 8 && p.splits <= 32 &&
                             2 * ((p.splits + 7) / 8) < (rows_per_cta + 2) / 3;
      KernelTimer kt("unembed_merge_sm103", a.stream);
      e = launch_pdl(many_rows ? unembed_merge_sm103<true> : unembed_merge_sm103<false>,
                     dim3(units, (unsigned)((total + cpc - 1) / cpc)), dim3(UM_THREADS), UM_SMEM,
                     a.stream, tm_wuv, tm_pieces, up);
      if (e != cudaSuccess) return e;
      return cudaGetLastError();
    }
  }
  {
    MergeParams mp{o_part, ml, a.lens, o_lat, R, p.chunk, p.splits, p.B * R,
                   a.topk ? a.topk_k : 0};
    KernelTimer kt("merge_sm103", a.stream);
    if (p.splits >= 48)
      e = launch_pdl(merge_sm103<1, 8>, dim3(p.B * R, 2), dim3(256), 0, a.stream, mp);
    else if (p.splits >= 32)
      e = launch_pdl(merge_sm103<1, 4>, dim3(p.B * R, 2), dim3(128), 0, a.stream, mp);
    else if (p.splits >= 16)
      e = launch_pdl(merge_sm103<2, 4>, dim3(p.B * R, 1), dim3(128), 0, a.stream, mp);
    else
      e = launch_pdl(merge_rows_sm103, dim3((p.B * R + MR_ROWS - 1) / MR_ROWS), dim3(32 * MR_ROWS),
                     0, a.stream, mp);
    if (e != cudaSuccess) return e;
  }
  {
    GemmParams gp{(__nv_bfloat16*)a.out, BL, p.H, kLat, p.v, NBu, 0, 0};
    KernelTimer kt("unembed_sm103", a.stream);
    e = launch_pdl(swapab_gemm_sm103, dim3(p.v / 128, p.H, (BL + NBu - 1) / NBu), dim3(128),
                   gemm_smem(kLat, NBu), a.stream, tm_wuv, tm_ol, gp);
    if (e != cudaSuccess) return e;
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
