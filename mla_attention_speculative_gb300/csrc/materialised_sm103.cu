// Materialised-branch MLA verify on GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// "One guard, 110x off the verify step", section "The defect": expand the
// whole cached latent back into full keys and values, then attend normally.
// Two kernels, bf16 operands with fp32 accumulation in tensor memory, chained
// with programmatic dependent launch:
//
//  expand_sm103    K_nope[b,h,t,:] = c_kv[b,t] . W_UK[h]^T   (512 -> n)
//                  V[b,h,t,:]      = c_kv[b,t] . W_UV[h]     (512 -> v)
//                  into one [B*H, Tmax, n+v] bf16 buffer (each head's keys and
//                  values contiguous).  One CTA per (128 cached positions,
//                  head) computes both products (n+v <= 256: two TMEM
//                  accumulators fed by each 64-wide latent chunk) or one of
//                  them (wider heads), two CTAs per SM; the chunks stream
//                  through a TMA ring; the bf16 tile leaves through shared
//                  memory with TMA stores clipped at Tmax.
//  mat_attn_sm103  causal attention of the L verify rows of one head against
//                  keys [K_nope || k_rope] (the RoPE key is shared by all heads)
//                  and values V: S = Q K^T on the tensor cores, an online
//                  softmax in registers (two threads per query row, each half
//                  of the tile's positions; the running max moved only when it
//                  grows by more than 2^8), P written back to tensor memory as
//                  the A operand of O += P V.  One CTA per (128-row query tile,
//                  head, sequence).
//
// Every wait is bounded; a wait that runs out sets the status word and the
// kernel finishes without waiting further (results are then undefined and
// mla_device_status reports MLA_ERR_TIMEOUT).

#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <mutex>
#include <utility>

#include "mla_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace mla {
using namespace sm103;

static __device__ int g_materialised_status;

namespace {

constexpr int kLat = 512;
constexpr int kSmemPerBlock = 232448;   // opt-in maximum per CTA
constexpr int kSmemPerSM = 233472;
constexpr int kSmemReserved = 1024;     // per CTA, taken by the runtime
constexpr int kSmemExtra = 1024 + 256;  // 1024-byte realignment + barriers
constexpr int kMatRowBytes = 2 * 128 * 4;  // per (warpgroup, row) floats of mat_attn

// The first 1024-byte boundary at or after the dynamic shared array, as an
// offset from the array itself (no integer round trip), so that the compiler
// still knows every pointer derived from it is a shared-memory one.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (sm103::smem_u32(p) & 1023u)) & 1023u);
}
__device__ __forceinline__ void report_timeout(int code) {
  atomicCAS(&g_materialised_status, 0, code);
}
__device__ __forceinline__ void wait_or_fail(bool& ok, uint32_t bar, uint32_t parity, int code) {
  if (!ok) return;
  if (!mbar_wait(bar, parity)) {
    ok = false;
    report_timeout(code);
  }
}

// Row of cached position t of sequence b in the 2-D cache tensors.  A page id
// outside [0, num_pages) forms no address: it is reported and the row becomes
// a wholly negative one, whose boxes TMA fills with zeros.
__device__ __forceinline__ int cache_y(const int32_t* page_table, int page_size, int max_pages,
                                       int num_pages, long long seq_stride, int b, int t) {
  if (page_table == nullptr) return (int)((long long)b * seq_stride + t);
  const int page = page_table[(long long)b * max_pages + t / page_size];
  if (page < 0 || page >= num_pages) {
    report_timeout(kBadPageSite);
    return -256;
  }
  return (int)((long long)page * page_size + (t % page_size));
}

// =========================================================================
// expansion GEMM
// =========================================================================
struct ExpandParams {
  const int32_t* lens;
  const int32_t* page_table;
  int page_size, max_pages, num_pages;
  long long seq_stride;
  int H, n, v, stages;
  uint32_t tmem_cols, v_col;  // TMEM allocation; V accumulator's first column
  int split;                  // 1: K_nope and V in separate CTAs (blockIdx.x & 1)
};

constexpr int EX_BM = 128;

__host__ __device__ constexpr int expand_stage_bytes(int n, int v) {
  return EX_BM * 128 + (n + v) * 128;
}

__global__ void __launch_bounds__(128, 1) expand_sm103(const __grid_constant__ CUtensorMap tm_ckv,
                                                       const __grid_constant__ CUtensorMap tm_wuk,
                                                       const __grid_constant__ CUtensorMap tm_wuv,
                                                       const __grid_constant__ CUtensorMap tm_out,
                                                       ExpandParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int mt = p.split ? blockIdx.x >> 1 : blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  // which products this CTA computes: both, or (split) K_nope or V alone
  const bool has_k = !p.split || (blockIdx.x & 1) == 0;
  const bool has_v = !p.split || (blockIdx.x & 1) == 1;
  pdl_wait();  // the cache and its lengths may come from the preceding kernel
  const int T = p.lens[b];
  const int t0 = mt * EX_BM;
  if (t0 >= T) return;
  const int n = p.n, v = p.v, S = p.stages;
  const int nk = has_k ? n : 0, nv = has_v ? v : 0;   // B columns of each product
  const uint32_t vcol = has_k ? p.v_col : 0u;         // V accumulator's TMEM column
  const int out0 = has_k ? 0 : n;                     // first output column
  const int SB = EX_BM * 128 + (nk + nv) * 128;
  uint64_t* bars = (uint64_t*)(smem + S * SB);  // [0,S) full, [S,2S) empty, 2S done
  uint32_t* slot = (uint32_t*)(bars + 2 * S + 1);
  volatile int* fail = (volatile int*)(slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[S + s]); };
  const uint32_t done = smem_u32(&bars[2 * S]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *fail = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  constexpr int kChunks = kLat / 64;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    // The 128-row cache tile is two 64-row boxes; with paging each box lies
    // in one page (page sizes are multiples of 64).  Rows at or past T are
    // loaded but never read back.
    bool ok = true;
    const int y0 = cache_y(p.page_table, p.page_size, p.max_pages, p.num_pages, p.seq_stride, b, t0);
    const int y1 = t0 + 64 < T
                       ? cache_y(p.page_table, p.page_size, p.max_pages, p.num_pages, p.seq_stride, b, t0 + 64)
                       : y0 + 64;
    int issued = 0;
    for (int kc = 0; kc < kChunks; ++kc) {
      const int s = kc % S;
      if (kc >= S) wait_or_fail(ok, empty(s), ((kc / S) - 1) & 1, 40);
      if (!ok) break;
      const uint32_t st = sbase + s * SB;
      mbar_arrive_expect_tx(full(s), SB);
      tma_load_2d(st, &tm_ckv, full(s), 64 * kc, y0);
      tma_load_2d(st + 8192, &tm_ckv, full(s), 64 * kc, y1);
      const uint32_t bn = st + EX_BM * 128;
      for (int r = 0; r < nk / 64; ++r)
        tma_load_2d(bn + r * 8192, &tm_wuk, full(s), 64 * kc, h * n + 64 * r);
      const uint32_t bv = bn + nk * 128;
      for (int j = 0; j < nv / 64; ++j)
        tma_load_2d(bv + j * 8192, &tm_wuv, full(s), 64 * j, h * kLat + 64 * kc);
      issued = kc + 1;
    }
    // no load may still be landing when the ring is reused for the output
    for (int kc = max(issued - S, 0); kc < issued; ++kc) mbar_wait(full(kc % S), (kc / S) & 1);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------- MMA
    bool ok = true;
    const uint32_t id_n = idesc_bf16(128, n, 0, 0);
    const uint32_t id_v = idesc_bf16(128, v, 0, 1);
    for (int kc = 0; kc < kChunks; ++kc) {
      const int s = kc % S;
      wait_or_fail(ok, full(s), (kc / S) & 1, 41);
      if (!ok) break;
      tc_fence_after();
      const uint32_t st = sbase + s * SB;
      const uint64_t da = sdesc_sw128(st, 16, 1024);
      const uint64_t dn = sdesc_sw128(st + EX_BM * 128, 16, 1024);
      const uint64_t dv = sdesc_sw128(st + EX_BM * 128 + nk * 128, 8192, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (has_k) mma_bf16(tmem, da + 2 * ks, dn + 2 * ks, id_n, (kc | ks) != 0);
        if (has_v) mma_bf16(tmem + vcol, da + 2 * ks, dv + 128 * ks, id_v, (kc | ks) != 0);
      }
      mma_commit(empty(s));
    }
    if (!ok) *fail = 1;
    mma_commit(done);
    if (!mbar_wait(done, 0)) {
      *fail = 1;
      report_timeout(42);
    }
  }
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  const bool ok = !*fail;
  if (ok) {
    // TMEM -> bf16 -> shared memory in the 128-byte-swizzled layout of the
    // store boxes (64 columns x 128 rows, 16 KB each, box 0 = output column
    // out0), then TMA stores.
    const int q = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    auto emit = [&](uint32_t col0, int width, int out_col0) {
      for (int c = 0; c < width; c += 32) {
        uint32_t r[32];
        tmem_ld16(tmem + lane_base + col0 + c, *(uint32_t(*)[16])(r));
        tmem_ld16(tmem + lane_base + col0 + c + 16, *(uint32_t(*)[16])(r + 16));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const int col = out_col0 - out0 + c + e;
          const uint32_t addr = sbase + (col >> 6) * (EX_BM * 128) + q * 128 +
                                ((((col & 63) >> 3) ^ (q & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                       "r"(pack_bf16(__uint_as_float(r[e]), __uint_as_float(r[e + 1]))),
                       "r"(pack_bf16(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]))),
                       "r"(pack_bf16(__uint_as_float(r[e + 4]), __uint_as_float(r[e + 5]))),
                       "r"(pack_bf16(__uint_as_float(r[e + 6]), __uint_as_float(r[e + 7])))
                       : "memory");
        }
      }
    };
    if (has_k) emit(0, n, 0);
    if (has_v) emit(vcol, v, n);
    fence_async_shared();
  }
  __syncthreads();
  if (ok && threadIdx.x == 0) {
    const int plane = b * p.H + h;
    for (int c = 0; c < (nk + nv) / 64; ++c)
      tma_store_3d(&tm_out, sbase + c * (EX_BM * 128), out0 + 64 * c, t0, plane);
    bulk_commit();
    // shared memory is free once the stores have read it; their writes are
    // complete when the grid is (the attention reads them after its wait)
    bulk_wait_read();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// =========================================================================
// flash attention over the expanded cache
// =========================================================================
struct MatAttnParams {
  const int32_t* lens;
  const int32_t* page_table;
  int page_size, max_pages, num_pages;
  long long seq_stride;
  __nv_bfloat16* out;  // [B, L, H, v]
  int L, H, n, v;
  int ks, vs;          // K ring and V ring depths
  float sl2;           // softmax scale x log2(e)
  int B;
  // split-KV when the query tiles alone leave SMs idle: each piece of a
  // query tile leaves O / l (bf16) and (m, l) for mat_combine_sm103
  int splits, chunk_tiles;
  // piece 0 covers KV tiles [0, first_tiles), piece sp >= 1 covers
  // [first_tiles + (sp - 1) * chunk_tiles, + chunk_tiles); first_tiles =
  // chunk_tiles unless one long and one short piece fill a partial wave
  int first_tiles;
  int sp_outer;  // 1: pieces slowest in the launch order (every long piece first)
  __nv_bfloat16* o_part;  // [B, splits, L, H, v]
  float* ml;              // [B, splits, L, H, 2]
};

constexpr int MA_BM = 128;
constexpr int MA_BN = 64;
constexpr int MA_NWG = 2;                       // softmax warpgroups; each takes half a row
constexpr int MA_CPT = MA_BN / MA_NWG;          // score columns per softmax thread
constexpr int MA_SOFTMAX = 128 * MA_NWG;
// warps: key producer, score-MMA issuer, value producer, P.V issuer, softmax
constexpr int MA_THREADS = 128 + MA_SOFTMAX;
constexpr uint32_t MA_TM_S = 256;  // S / P buffers at 256 + 64*sb; O at [0, v)
constexpr int MA_SBUF = 4;         // S / P buffers (TMEM columns 256..511)

__host__ __device__ constexpr int mat_q_bytes(int n) { return (n / 64 + 1) * MA_BM * 128; }
// A key tile [K_nope || k_rope] (64 positions) and a value tile, in 64-column chunks.
__host__ __device__ constexpr int mat_k_bytes(int n) { return (n / 64 + 1) * MA_BN * 128; }
__host__ __device__ constexpr int mat_v_bytes(int v) { return (v / 64) * MA_BN * 128; }

// barriers: Q, then one S full, P full and O done per S buffer (tile i uses
// copy i % MA_SBUF, phase i / MA_SBUF), drain x2 (one per MMA issuer), then the
// K ring (full, empty) and the V ring (full, empty)
enum {
  M_QFULL = 0,
  M_SFULL = 1,
  M_PFULL = M_SFULL + MA_SBUF,
  M_ODONE = M_PFULL + MA_SBUF,
  M_DRAIN = M_ODONE + MA_SBUF,
  M_RINGS = M_DRAIN + 2
};

// NQ = n/64 + 1 (the 64-column chunks of [q_nope || q_rope]) is a template
// parameter so the score MMAs unroll with constant descriptor offsets: tcgen05
// MMA issue is nearly synchronous, so arithmetic between MMAs idles the pipe.
template <int NQ>
__global__ void __launch_bounds__(MA_THREADS, 1) mat_attn_sm103(const __grid_constant__ CUtensorMap tm_qn,
                                                         const __grid_constant__ CUtensorMap tm_qr,
                                                         const __grid_constant__ CUtensorMap tm_kx,
                                                         const __grid_constant__ CUtensorMap tm_kr,
                                                         MatAttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // One CTA per (128-row query tile, KV piece, head, sequence), the query
  // tiles and pieces of one head next to each other so that they share its
  // expanded keys and values in L2.  (Handing out the longest query tiles
  // first instead made the causal prefill 8 % slower: every wave then read
  // 152 heads' keys and values.)
  const int nqt = (p.L + MA_BM - 1) / MA_BM;
  const int qt = (int)(blockIdx.x % nqt);
  const int rest = (int)(blockIdx.x / nqt);
  int sp, h, b;
  if (p.sp_outer) {
    h = rest % p.H;
    b = (rest / p.H) % p.B;
    sp = rest / (p.H * p.B);
  } else {
    sp = rest % p.splits;
    h = (rest / p.splits) % p.H;
    b = rest / (p.splits * p.H);
  }
  const int T = p.lens[b];
  const int n = p.n, v = p.v, L = p.L;
  const int l0 = qt * MA_BM;
  const int l_last = min(L - 1, l0 + MA_BM - 1);
  const int kv_end = T - L + l_last + 1;  // no row of the tile sees t >= kv_end
  // this CTA's KV tiles: [i0, i0 + ntiles) of the tile's visible ones; the
  // loops below count from 0, positions add tbase
  const int i0 = sp == 0 ? 0 : p.first_tiles + (sp - 1) * p.chunk_tiles;
  const int ntiles = min((kv_end + MA_BN - 1) / MA_BN - i0, sp == 0 ? p.first_tiles : p.chunk_tiles);
  const int tbase = i0 * MA_BN;
  if (ntiles <= 0) {
    // a piece past what the tile sees: an empty part for the combine
    for (int q = threadIdx.x; q < MA_BM; q += blockDim.x) {
      if (l0 + q >= L) continue;
      const size_t prow = (((size_t)b * p.splits + sp) * L + l0 + q) * p.H + h;
      p.ml[prow * 2] = -FLT_MAX;
      p.ml[prow * 2 + 1] = 0.f;
    }
    return;
  }
  const int KS = p.ks, VS = p.vs;
  const int QB = mat_q_bytes(n), KB = mat_k_bytes(n), VB = mat_v_bytes(v);
  const uint32_t sQ = smem_u32(smem), sK = sQ + QB, sV = sK + KS * KB;
  uint8_t* tail = smem + QB + KS * KB + VS * VB;
  uint64_t* bars = (uint64_t*)tail;
  uint32_t* slot = (uint32_t*)(bars + M_RINGS + 2 * KS + 2 * VS);
  // per (warpgroup, row): the tile maxima, and at the end the row sums
  float* xrow = (float*)(tail + 256);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto k_full = [&](int s) { return bar(M_RINGS + s); };
  auto k_empty = [&](int s) { return bar(M_RINGS + KS + s); };
  auto v_full = [&](int s) { return bar(M_RINGS + 2 * KS + s); };
  auto v_empty = [&](int s) { return bar(M_RINGS + 2 * KS + VS + s); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(M_QFULL), 1);
    for (int i = 0; i < MA_SBUF; ++i) {
      mbar_init(bar(M_SFULL + i), 1);
      mbar_init(bar(M_PFULL + i), MA_SOFTMAX);
      mbar_init(bar(M_ODONE + i), 1);
    }
    mbar_init(bar(M_DRAIN), 1);
    mbar_init(bar(M_DRAIN + 1), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int plane = b * p.H + h;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // Warp 0 loads Q and the key ring, warp 2 the value ring (each in its own
    // warp, so neither waits behind the other): a key tile is free once S has
    // read it, a value tile once P.V has.
    if (lane == 0) {
      bool ok = true;
      pdl_wait();  // the expanded cache comes from the expansion kernel
      const int qrow = b * L + l0;
      mbar_arrive_expect_tx(bar(M_QFULL), QB);
      for (int c = 0; c < n / 64; ++c)
        tma_load_2d(sQ + c * MA_BM * 128, &tm_qn, bar(M_QFULL), h * n + 64 * c, qrow);
      tma_load_2d(sQ + (n / 64) * MA_BM * 128, &tm_qr, bar(M_QFULL), h * 64, qrow);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % KS;
        if (i >= KS) wait_or_fail(ok, k_empty(s), ((i / KS) - 1) & 1, 50);
        if (!ok) break;
        const int t0 = tbase + i * MA_BN;
        const int y = cache_y(p.page_table, p.page_size, p.max_pages, p.num_pages, p.seq_stride, b, t0);
        const uint32_t st = sK + s * KB;
        mbar_arrive_expect_tx(k_full(s), KB);
        for (int c = 0; c < n / 64; ++c)
          tma_load_3d(st + c * 8192, &tm_kx, k_full(s), 64 * c, t0, plane);
        tma_load_2d(st + (n / 64) * 8192, &tm_kr, k_full(s), 0, y);
        issued = i + 1;
      }
      // drain: nothing may still be landing when the CTA exits
      mbar_wait(bar(M_QFULL), 0);
      for (int i = max(issued - KS, 0); i < issued; ++i) mbar_wait(k_full(i % KS), (i / KS) & 1);
    }
  } else if (warp == 2) {
    if (lane == 0) {
      bool ok = true;
      pdl_wait();
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % VS;
        if (i >= VS) wait_or_fail(ok, v_empty(s), ((i / VS) - 1) & 1, 57);
        if (!ok) break;
        const uint32_t st = sV + s * VB;
        mbar_arrive_expect_tx(v_full(s), VB);
        for (int j = 0; j < v / 64; ++j)
          tma_load_3d(st + j * 8192, &tm_kx, v_full(s), n + 64 * j, tbase + i * MA_BN, plane);
        issued = i + 1;
      }
      for (int i = max(issued - VS, 0); i < issued; ++i) mbar_wait(v_full(i % VS), (i / VS) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- score-MMA issuer
    // S(i) goes to S buffer i % MA_SBUF, which holds P(i - MA_SBUF) until its
    // P.V is done.
    // MMA issue is nearly synchronous, so the scores and P.V come from two
    // warps: a wait in one leaves the tensor pipe to the other.
    if (lane == 0) {
      bool ok = true;
      const uint64_t dq = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk = sdesc_sw128(sK, 16, 1024);
      const uint32_t id_s = idesc_bf16(MA_BM, MA_BN, 0, 0);
      wait_or_fail(ok, bar(M_QFULL), 0, 51);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int s = i % KS, sb = i % MA_SBUF;
        wait_or_fail(ok, k_full(s), (i / KS) & 1, 52);
        // S buffer sb held P(i - MA_SBUF): its P.V must be done
        if (i >= MA_SBUF) wait_or_fail(ok, bar(M_ODONE + sb), ((i / MA_SBUF) - 1) & 1, 60);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dks = dk + (uint64_t)(s * (KB >> 4));
        const uint32_t dst = tmem + MA_TM_S + sb * MA_BN;
#pragma unroll
        for (int c = 0; c < NQ; ++c)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(dst, dq + ((c * MA_BM * 128 + ks * 32) >> 4),
                     dks + ((c * 8192 + ks * 32) >> 4), id_s, (c | ks) != 0);
        mma_commit(bar(M_SFULL + sb));
        mma_commit(k_empty(s));
      }
      mma_commit(bar(M_DRAIN));
      mbar_wait(bar(M_DRAIN), 0);
    }
  } else if (warp == 3) {
    // --------------------------------------------------------- P.V issuer
    if (lane == 0) {
      bool ok = true;
      const uint64_t dv = sdesc_sw128(sV, 8192, 1024);
      const uint32_t id_o = idesc_bf16(MA_BM, v, 0, 1);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int vj = j % VS, pb = j % MA_SBUF;
        wait_or_fail(ok, bar(M_PFULL + pb), (j / MA_SBUF) & 1, 53);
        wait_or_fail(ok, v_full(vj), (j / VS) & 1, 58);
        if (!ok) break;
        tc_fence_after();
        const uint64_t voff = (uint64_t)(vj * (VB >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_tmem_a(tmem, tmem + MA_TM_S + pb * MA_BN + ks * 8, dv + voff + ks * 128, id_o,
                          (j > 0 || ks > 0));
        mma_commit(bar(M_ODONE + pb));
        mma_commit(v_empty(vj));
      }
      mma_commit(bar(M_DRAIN + 1));
      mbar_wait(bar(M_DRAIN + 1), 0);
    }
  } else {
    // ------------------------------------------------- softmax warpgroups
    // Thread (wg, q) owns row q, score columns MA_CPT*wg.. of each tile and O
    // columns (v/MA_NWG)*wg..; the warpgroups combine their row maxima (and at
    // the end their row sums) through shared memory.
    const int wg = (warp - 4) >> 2;
    const int q = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const int c0 = MA_CPT * wg;
    const int opt = v / MA_NWG;            // O columns per thread
    const int sm_tid = threadIdx.x - 128;
    const int l = min(l0 + q, L - 1);
    const int last_t = T - L + l;          // the last position row l may see
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    for (int i = 0; i < ntiles; ++i) {
      const int sb = i % MA_SBUF;
      const int t0 = tbase + i * MA_BN;
      wait_or_fail(ok, bar(M_SFULL + sb), (i / MA_SBUF) & 1, 54);
      tc_fence_after();
      uint32_t u[MA_CPT];
#pragma unroll
      for (int k = 0; k < MA_CPT / 16; ++k)
        tmem_ld16(tmem + lane_base + MA_TM_S + sb * MA_BN + c0 + 16 * k,
                  *(uint32_t(*)[16])(u + 16 * k));
      tmem_wait_ld();
      // Masked columns: past the row's causal limit (this also covers
      // positions at or past T, whose keys may hold anything).
      float s[MA_CPT];
      const bool edge = t0 + MA_BN - 1 > T - L;
#pragma unroll
      for (int j = 0; j < MA_CPT; ++j) {
        const float x = __uint_as_float(u[j]) * p.sl2;
        s[j] = (!edge || t0 + c0 + j <= last_t) ? x : -INFINITY;
      }
      float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int j = 4; j < MA_CPT; ++j) m4[j & 3] = fmaxf(m4[j & 3], s[j]);
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      xrow[wg * MA_BM + q] = mt;
      named_bar_sync(1, MA_SOFTMAX);
#pragma unroll
      for (int g = 0; g < MA_NWG; ++g) mt = fmaxf(mt, xrow[g * MA_BM + q]);
      // every warpgroup has read this tile's maxima before any writes the next
      named_bar_sync(2, MA_SOFTMAX);
      const bool need = mt > m_run + 8.f;
      const float m_new = need ? mt : m_run;
      const float factor = need ? ex2(m_run - m_new) : 1.f;
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        // O must hold P(i-1) V(i-1) before it is rescaled
        wait_or_fail(ok, bar(M_ODONE + (i - 1) % MA_SBUF), ((i - 1) / MA_SBUF) & 1, 55);
        tc_fence_after();
        for (int c = 0; c < opt; c += 16) {
          uint32_t w[16];
          tmem_ld16(tmem + lane_base + opt * wg + c, w);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * factor);
          tmem_st16(tmem + lane_base + opt * wg + c, w);
        }
      }
      l_run *= factor;
      m_run = m_new;
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pk[MA_CPT / 2];
#pragma unroll
      for (int e = 0; e < MA_CPT / 2; ++e) {
        const float a = ex2(s[2 * e] - m_use);
        const float d = ex2(s[2 * e + 1] - m_use);
        rs0 += a;
        rs1 += d;
        pk[e] = pack_bf16(a, d);
      }
      l_run += rs0 + rs1;
      // P(i) as bf16 pairs over S buffer sb: this thread's positions are the
      // pair columns c0/2 ..
#pragma unroll
      for (int k = 0; k < MA_CPT / 32; ++k)
        tmem_st16(tmem + lane_base + MA_TM_S + sb * MA_BN + c0 / 2 + 16 * k,
                  *(const uint32_t(*)[16])(pk + 16 * k));
      // Value rows at or past T in the last tile may hold anything (0 x NaN
      // would poison O): zero them in shared memory before P V reads them.
      if (ok && t0 + MA_BN > T) {
        const int z0 = max(T - t0, 0);
        wait_or_fail(ok, v_full(i % VS), (i / VS) & 1, 59);  // the value tile has landed
        const uint32_t st = sV + (i % VS) * VB;
        const int units = (MA_BN - z0) * 8;  // 16-byte units per 64-column chunk
        for (int w = sm_tid; w < (v / 64) * units; w += MA_SOFTMAX) {
          const int c = w / units, r = w - c * units;
          const uint32_t addr = st + c * 8192 + (z0 + r / 8) * 128 + (r & 7) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                       : "memory");
        }
        fence_async_shared();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(M_PFULL + sb));
    }
    // ---------------------------------------------------------------- epilogue
    wait_or_fail(ok, bar(M_ODONE + (ntiles - 1) % MA_SBUF), ((ntiles - 1) / MA_SBUF) & 1, 56);
    tc_fence_after();
    pdl_launch_dependents();
    xrow[wg * MA_BM + q] = l_run;
    named_bar_sync(1, MA_SOFTMAX);
    float l_tot = 0.f;
#pragma unroll
    for (int g = 0; g < MA_NWG; ++g) l_tot += xrow[g * MA_BM + q];
    const bool live = l0 + q < L;
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    // one piece: the output row; several: this piece's O / l and (m, l)
    const size_t orow = p.splits > 1
                            ? (((size_t)b * p.splits + sp) * L + (live ? l0 + q : 0)) * p.H + h
                            : ((size_t)b * L + (live ? l0 + q : 0)) * p.H + h;
    __nv_bfloat16* dst = (p.splits > 1 ? p.o_part : p.out) + orow * (size_t)v + opt * wg;
    if (p.splits > 1 && live && wg == 0) {
      p.ml[orow * 2] = m_run == -INFINITY ? -FLT_MAX : m_run;
      p.ml[orow * 2 + 1] = l_tot;
    }
    for (int c = 0; c < opt; c += 32) {
      uint32_t r[32];
      tmem_ld16(tmem + lane_base + opt * wg + c, *(uint32_t(*)[16])(r));
      tmem_ld16(tmem + lane_base + opt * wg + c + 16, *(uint32_t(*)[16])(r + 16));
      tmem_wait_ld();
      if (live) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(r[e + 4]) * inv, __uint_as_float(r[e + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(r[e + 6]) * inv, __uint_as_float(r[e + 7]) * inv);
          *(uint4*)(dst + c + e) = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// out[b, l, h, :] = sum_s w_s (O_s / l_s)[b, l, h, :] / sum_s w_s with
// w_s = 2^(m_s - M) l_s over the KV pieces of the materialised attention (M
// the largest m_s; empty pieces have l_s = 0).  One warp per output row; a
// lane holds one piece's (m, l) and 8 columns of the sums.
constexpr int MC_ROWS = 4;  // rows (warps) per CTA
__global__ void __launch_bounds__(32 * MC_ROWS)
    mat_combine_sm103(const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ ml,
                      __nv_bfloat16* __restrict__ out, int rows, int LH, int v, int splits) {
  pdl_wait();  // the pieces come from the attention
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * MC_ROWS + warp;
  if (row >= rows) return;
  const int b = row / LH, r = row - b * LH;
  // the first columns' piece loads go out before the weights are known: they
  // do not depend on them (an empty piece is read, never added)
  const int c0 = lane * 8;
  uint4 x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < splits && c0 < v)
      x[j] = *(const uint4*)(o_part + (((size_t)b * splits + j) * LH + r) * v + c0);
  float2 e = make_float2(-FLT_MAX, 0.f);
  if (lane < splits) e = *(const float2*)(ml + (((size_t)b * splits + lane) * LH + r) * 2);
  float M = e.y > 0.f ? e.x : -FLT_MAX;
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = e.y > 0.f ? ex2(e.x - M) * e.y : 0.f;
  float den = w;
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  for (int c = c0; c < v; c += 256) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < splits; s0 += 4) {
      // up to four pieces' loads in flight before any of them is used
      if (c != c0 || s0 != 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (s0 + j < splits)
            x[j] = *(const uint4*)(o_part + (((size_t)b * splits + s0 + j) * LH + r) * v + c);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (s0 + j >= splits) break;
        const float ws = __shfl_sync(0xffffffffu, w, s0 + j);
        if (ws == 0.f) continue;
        const uint32_t u[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[2 * k] = fmaf(ws, __uint_as_float(u[k] << 16), acc[2 * k]);
          acc[2 * k + 1] = fmaf(ws, __uint_as_float(u[k] & 0xffff0000u), acc[2 * k + 1]);
        }
      }
    }
    *(uint4*)(out + (size_t)row * v + c) =
        make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                   pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
  }
}

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

// Expansion layout.  When n + v <= 256 one CTA computes both products (two
// accumulators in 256 TMEM columns) and two CTAs share an SM.  Otherwise
// K_nope and V get separate CTAs (each <= 256 columns, the latent tile read
// once per product), again two per SM, so one CTA's epilogue overlaps the
// other's GEMM.  The ring gets half the SM's shared memory either way.
struct ExpandShape {
  uint32_t tmem_cols, v_col;
  int stages, smem, split;
};
ExpandShape expand_shape(int n, int v) {
  ExpandShape e;
  e.split = n + v > 256 ? 1 : 0;
  e.tmem_cols = 256u;
  e.v_col = e.split ? 0u : (uint32_t)n;
  const int budget = kSmemPerSM / 2 - kSmemReserved;
  const int sb = e.split ? EX_BM * 128 + (n > v ? n : v) * 128 : expand_stage_bytes(n, v);
  int s = (budget - kSmemExtra) / sb;
  e.stages = s > 4 ? 4 : s;
  e.smem = e.stages * sb + kSmemExtra;
  return e;
}
// Key and value ring depths that fit next to Q, or {0, 0} if not even two of
// each fit.  Values come first: a key tile is freed as soon as S has read it,
// a value tile only after P.V, so the value ring is the one that runs dry.
struct MatRings {
  int ks, vs, smem;
};
MatRings mat_rings(int n, int v) {
  const int budget = kSmemPerBlock - kSmemExtra - kMatRowBytes - mat_q_bytes(n);
  const int cand[][2] = {{4, 4}, {4, 3}, {3, 4}, {3, 3}, {4, 2}, {3, 2}, {2, 4}, {2, 3}, {2, 2}};
  for (const auto& c : cand) {
    const int bytes = c[0] * mat_k_bytes(n) + c[1] * mat_v_bytes(v);
    if (bytes <= budget)
      return {c[0], c[1], mat_q_bytes(n) + bytes + kSmemExtra + kMatRowBytes};
  }
  return {0, 0, 0};
}

}  // namespace

bool fast_materialised_supported(const Plan& p) {
  if (!(p.dtype == MLA_DTYPE_BF16 && p.r == kLat && p.rope == 64 && p.n % 64 == 0 && p.n >= 64 &&
        p.n <= 256 && p.v % 64 == 0 && p.v >= 64 && p.v <= 256))
    return false;
  const ExpandShape e = expand_shape(p.n, p.v);
  // the output tile (128 rows x the CTA's columns, bf16) is staged in the drained ring
  const int cols = e.split ? (p.n > p.v ? p.n : p.v) : p.n + p.v;
  return e.stages >= 2 && e.smem - kSmemExtra >= EX_BM * cols * 2 && mat_rings(p.n, p.v).ks >= 2;
}

namespace {

// KV pieces per query tile of the materialised attention: when the (query
// tile, head, sequence) CTAs leave SMs idle, each is cut into pieces of
// chunk_tiles KV tiles, choosing the cut that minimises waves x (tiles per
// piece + the fixed cost of a CTA, about four tiles) with one CTA per SM.
struct MatSplit {
  int splits = 1, chunk_tiles = 1, first_tiles = 1, sp_outer = 0;
};
MatSplit mat_split(const Plan& p) {
  const long long units = (long long)((p.L + MA_BM - 1) / MA_BM) * p.H * p.B;
  const int tiles = (p.Tmax + MA_BN - 1) / MA_BN;
  const long long slots = device_sm_count();
  MatSplit best;
  best.chunk_tiles = tiles;
  const long long whole = ((units + slots - 1) / slots) * (tiles + 4);
  long long best_cost = whole;
  for (int s = 2; s <= 16; ++s) {
    const int ct = (tiles + s - 1) / s;
    if (ct < 8) break;
    const long long cost = ((units * s + slots - 1) / slots) * (ct + 4);
    if (cost < best_cost) {
      best_cost = cost;
      best.chunk_tiles = ct;
    }
  }
  // the pieces' round trip and the combine kernel cost more than the model's
  // four tiles: cut only for a clear gain (measured: four pieces of the
  // 512/192/256 L = 1024 call at T = 8192 by the model's 5 % were 8 % slower)
  if (best_cost * 4 > whole * 3) {
    best.chunk_tiles = tiles;
    best_cost = whole;
  }
  best.splits = (tiles + best.chunk_tiles - 1) / best.chunk_tiles;
  best.first_tiles = best.chunk_tiles;
  // A partial last wave leaves SMs idle.  Cut each unit into one long piece
  // of a >= tiles / 2 tiles and one short piece of the rest, long pieces
  // launched first: the long ones take W = ceil(units / slots) waves of
  // a + o, and the short ones (tiles - a + o each) run on the SMs the last
  // long wave leaves idle, any that do not fit there in further waves after.
  // Kept for a clear gain (10 % by the model; the combine kernel is one more
  // launch).
  const long long idle = (slots - units % slots) % slots;
  if (idle > 0 && tiles >= 16) {
    constexpr long long o = 4;
    const long long W = (units + slots - 1) / slots;
    long long best_a = 0, best_span = best_cost;
    for (long long a = (tiles + 1) / 2; a < tiles; ++a) {
      const long long piece = tiles - a + o;
      // short pieces that fit beside the last long wave: idle SMs, each
      // running a + o worth of them
      const long long fit = idle * ((a + o) / piece);
      const long long rest = units > fit ? units - fit : 0;
      const long long span = W * (a + o) + ((rest + slots - 1) / slots) * piece;
      if (span < best_span) {
        best_span = span;
        best_a = a;
      }
    }
    if (best_a > 0 && best_span * 10 <= best_cost * 9) {
      best.splits = 2;
      best.first_tiles = (int)best_a;
      best.chunk_tiles = tiles - (int)best_a;
      best.sp_outer = 1;
    }
  }
  return best;
}

size_t align256_bytes(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t fast_materialised_workspace(const Plan& p) {
  size_t bytes = align256_bytes((size_t)p.B * p.H * p.Tmax * (p.n + p.v) * 2);
  const MatSplit ms = mat_split(p);
  if (ms.splits > 1) {
    const size_t rows = (size_t)p.B * ms.splits * p.L * p.H;
    bytes += align256_bytes(rows * p.v * 2) + align256_bytes(rows * 2 * sizeof(float));
  }
  return bytes;
}

cudaError_t launch_fast_materialised(const Plan& p, const Args& a) {
  const CacheView& c = a.cache;
  const long long cache_rows = c.page_table ? (long long)c.num_pages * c.page_size
                                            : (long long)(p.B - 1) * c.seq_stride + p.Tmax;
  __nv_bfloat16* kexp = (__nv_bfloat16*)(a.ws + p.off_exp);
  const int d = p.n + p.v;
  const uint64_t planes = (uint64_t)p.B * p.H;
  CUtensorMap tm_ckv, tm_wuk, tm_wuv, tm_store, tm_qn, tm_qr, tm_kx, tm_kr;
  bool ok = make_tmap_bf16_2d(&tm_ckv, c.c_kv, kLat, cache_rows, c.ckv_stride * 2, 64, 64, 128);
  ok = ok && make_tmap_bf16_2d(&tm_wuk, a.W_UK, kLat, (uint64_t)p.H * p.n, kLat * 2, 64, 64, 128);
  ok = ok && make_tmap_bf16_2d(&tm_wuv, a.W_UV, p.v, (uint64_t)p.H * kLat, (uint64_t)p.v * 2, 64,
                               64, 128);
  ok = ok && make_tmap_bf16_3d(&tm_store, kexp, d, p.Tmax, planes, (uint64_t)d * 2,
                               (uint64_t)p.Tmax * d * 2, 64, EX_BM);
  ok = ok && make_tmap_bf16_2d(&tm_qn, a.q_nope, (uint64_t)p.H * p.n, (uint64_t)p.B * p.L,
                               (uint64_t)p.H * p.n * 2, 64, MA_BM, 128);
  ok = ok && make_tmap_bf16_2d(&tm_qr, a.q_rope, (uint64_t)p.H * 64, (uint64_t)p.B * p.L,
                               (uint64_t)p.H * 64 * 2, 64, MA_BM, 128);
  ok = ok && make_tmap_bf16_3d(&tm_kx, kexp, d, p.Tmax, planes, (uint64_t)d * 2,
                               (uint64_t)p.Tmax * d * 2, 64, MA_BN);
  ok = ok && make_tmap_bf16_2d(&tm_kr, c.k_rope, 64, cache_rows, c.kr_stride * 2, 64, MA_BN, 128);
  if (!ok) return cudaErrorInvalidValue;

  const ExpandShape es = expand_shape(p.n, p.v);
  const MatRings mr = mat_rings(p.n, p.v);
  const int ma_smem = mr.smem;
  // shared-memory opt-in, once per device (calls may come from several threads)
  static std::mutex attrs_mu;
  static bool attrs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> attrs_lock(attrs_mu);
  if (dev >= 0 && dev < 64 && !attrs[dev]) {
    cudaError_t e = cudaFuncSetAttribute(expand_sm103, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemPerBlock);
    const void* attn[] = {(const void*)mat_attn_sm103<2>, (const void*)mat_attn_sm103<3>,
                          (const void*)mat_attn_sm103<4>, (const void*)mat_attn_sm103<5>};
    for (int k = 0; k < 4 && e == cudaSuccess; ++k)
      e = cudaFuncSetAttribute(attn[k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemPerBlock);
    if (e != cudaSuccess) return e;
    attrs[dev] = true;
  }
  cudaError_t e;
  {
    ExpandParams ep{a.lens, c.page_table, c.page_size, c.max_pages, c.num_pages, c.seq_stride,
                    p.H,    p.n,          p.v,         es.stages,   es.tmem_cols,
                    es.v_col, es.split};
    KernelTimer kt("expand_sm103", a.stream);
    const int mtiles = (p.Tmax + EX_BM - 1) / EX_BM;
    e = launch_pdl(expand_sm103, dim3(mtiles * (es.split ? 2 : 1), p.H, p.B), dim3(128), es.smem,
                   a.stream, tm_ckv, tm_wuk, tm_wuv, tm_store, ep);
    if (e != cudaSuccess) return e;
  }
  {
    const MatSplit ms = mat_split(p);
    char* ws_pieces = a.ws + p.off_exp +
                      align256_bytes((size_t)p.B * p.H * p.Tmax * (p.n + p.v) * 2);
    const size_t prow = (size_t)p.B * ms.splits * p.L * p.H;
    MatAttnParams mp{a.lens, c.page_table, c.page_size, c.max_pages, c.num_pages, c.seq_stride,
                     (__nv_bfloat16*)a.out, p.L, p.H, p.n, p.v, mr.ks, mr.vs,
                     p.scale * 1.4426950408889634f, p.B, ms.splits, ms.chunk_tiles,
                     ms.first_tiles, ms.sp_outer,
                     (__nv_bfloat16*)ws_pieces,
                     (float*)(ws_pieces + align256_bytes(prow * p.v * 2))};
    KernelTimer kt("mat_attn_sm103", a.stream);
    const dim3 grid((unsigned)(((p.L + MA_BM - 1) / MA_BM) * p.H * p.B * ms.splits));
    auto go = [&](auto kernel) {
      return launch_pdl(kernel, grid, dim3(MA_THREADS), ma_smem, a.stream, tm_qn, tm_qr, tm_kx,
                        tm_kr, mp);
    };
    switch (p.n / 64 + 1) {  // n is a multiple of 64 in [64, 256]
      case 2: e = go(mat_attn_sm103<2>); break;
      case 3: e = go(mat_attn_sm103<3>); break;
      case 4: e = go(mat_attn_sm103<4>); break;
      default: e = go(mat_attn_sm103<5>); break;
    }
    if (e != cudaSuccess) return e;
    if (ms.splits > 1) {
      const int rows = p.B * p.L * p.H;
      KernelTimer kc("mat_combine_sm103", a.stream);
      e = launch_pdl(mat_combine_sm103, dim3((rows + MC_ROWS - 1) / MC_ROWS), dim3(32 * MC_ROWS),
                     0, a.stream, (const __nv_bfloat16*)mp.o_part, (const float*)mp.ml,
                     (__nv_bfloat16*)a.out, rows, p.L * p.H, p.v, ms.splits);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

int materialised_device_status(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_materialised_status, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_materialised_status, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace mla
