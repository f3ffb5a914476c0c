// Speculative-rollback state maintenance on the GPU.
//
// "Over 107tok/s Qwen3.8-Flash-Next on M3 Ultra":
//  * section "A later extension: load snapshot history once", Algorithm 4
//    (recognise a safe snapshot group) and Algorithm 5 (one load per row,
//    then the concatenation and every snapshot window written from it):
//    mla_concat_snapshots.  Every source word is loaded once and the
//    concatenated row and each window's s words are written from that load.
//    For the contiguous row layouts a CTA stages 256 channels' words in
//    shared memory and writes X and the windows as contiguous runs; other
//    layouts give a thread one (channel, sequence) row in registers, as the
//    page does.  When the group is not safe to fuse, the ordinary path runs:
//    the concatenation, then one copy per window that reads it back.  Words
//    are moved as uint32 bit patterns.
//  * section "Keep the pooled keys; score them again", ValidBlock and
//    Algorithm 1 (retain a rollback-valid prefix): mla_rollback_valid_prefix.
//    The predicate is checked for every block in parallel and the prefix ends
//    at the first block that fails it (a minimum over the failing indices).

#include <algorithm>
#include <utility>
#include <vector>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kMaxWindows = 8;
constexpr int kMaxRow = 16;

struct Strides {
  long long i, h, q;
};
struct Window {
  int a;
  long long offset, stride;
};
struct ConcatParams {
  const uint32_t* S;
  const uint32_t* T;
  uint32_t* X;
  uint32_t* cache;
  Strides ss, ts, xs;
  int s, n, H, Q, k;
  int magic_w, magic_s;  // div_magic(s + n), div_magic(s)
  Window w[kMaxWindows];
};

// Algorithm 5 for any strides: one thread per row, 128 threads per CTA.
__global__ void __launch_bounds__(128) concat_snapshots_kernel(ConcatParams p) {
  const long long g = (long long)blockIdx.x * 128 + threadIdx.x;
  if (g >= (long long)p.H * p.Q) return;
  const int h = (int)(g % p.H), q = (int)(g / p.H);
  uint32_t v[kMaxRow];
#pragma unroll
  for (int i = 0; i < kMaxRow; ++i) {
    v[i] = 0u;
    if (i < p.s) v[i] = p.S[i * p.ss.i + h * p.ss.h + q * p.ss.q];
    else if (i < p.s + p.n) v[i] = p.T[(i - p.s) * p.ts.i + h * p.ts.h + q * p.ts.q];
  }
#pragma unroll
  for (int i = 0; i < kMaxRow; ++i)
    if (i < p.s + p.n) p.X[i * p.xs.i + h * p.xs.h + q * p.xs.q] = v[i];
  for (int j = 0; j < p.k; ++j) {
    uint32_t* d = p.cache + p.w[j].offset + q * p.w[j].stride + (long long)h * p.s;
    const int a = p.w[j].a;
#pragma unroll
    for (int i = 0; i < kMaxRow / 2; ++i) {
      if (i >= p.s) break;
      // V[a + i] with a register-resident array: select, never index
      uint32_t x = 0u;
#pragma unroll
      for (int t = 0; t < kMaxRow; ++t) x = (t == a + i) ? v[t] : x;
      d[i] = x;
    }
  }
}

// The same for the contiguous row layouts: S rows of s words and X rows of
// s + n words per channel, T rows of n words or channel-fastest planes.  A CTA
// takes 256 channels of one sequence: it loads their S and T words into
// shared memory in coalesced runs (each source word once), then writes their
// X rows and every window's s words per channel as contiguous runs, so no
// warp store is scattered over rows.
constexpr int kRowsPerCta = 256;

// Element e of a run of rows `w` words wide, walked 256 at a time: row and
// column advance by 256 / w and 256 % w with a carry, no division per word.
// The start uses e / w = (e * m) >> 16 with m = ceil(2^16 / w), exact for
// e < 4096 and w <= 16 (the error e (m - 2^16/w) / 2^16 < 1/16 <= 1/w).
__host__ __device__ constexpr int div_magic(int w) { return (65536 + w - 1) / w; }
struct RowWalk {
  int h, i, dq, dr, w;
  __device__ RowWalk(int e, int w_, int magic)
      : h((e * magic) >> 16), i(e - ((e * magic) >> 16) * w_), dq((kRowsPerCta * magic) >> 16),
        dr(kRowsPerCta - ((kRowsPerCta * magic) >> 16) * w_), w(w_) {}
  __device__ void next() {
    h += dq;
    i += dr;
    if (i >= w) {
      i -= w;
      ++h;
    }
  }
};

__global__ void __launch_bounds__(kRowsPerCta) concat_rows_kernel(ConcatParams p, int t_rows) {
  __shared__ uint32_t sS[kRowsPerCta * (kMaxRow / 2)];
  __shared__ uint32_t sT[kRowsPerCta * kMaxRow];
  const int q = blockIdx.y;
  const int h0 = blockIdx.x * kRowsPerCta;
  const int R = min(kRowsPerCta, p.H - h0);
  const int s = p.s, n = p.n, w = s + n;
  // every load of the thread is issued before the first store to shared memory
  const uint32_t* Sb = p.S + q * p.ss.q + (long long)h0 * s;
  uint32_t vs[kMaxRow / 2], vt[kMaxRow];
#pragma unroll
  for (int m = 0; m < kMaxRow / 2; ++m) {
    const int e = threadIdx.x + m * kRowsPerCta;
    vs[m] = e < R * s ? Sb[e] : 0u;
  }
  const uint32_t* Tb = p.T + q * p.ts.q + (t_rows ? (long long)h0 * n : (long long)h0);
#pragma unroll
  for (int m = 0; m < kMaxRow; ++m) {
    // row layout: word threadIdx + 256 m of the block; planes: plane m, channel threadIdx
    const bool live = t_rows ? threadIdx.x + m * kRowsPerCta < R * n
                             : m < n && (int)threadIdx.x < R;
    vt[m] = live ? Tb[t_rows ? threadIdx.x + m * kRowsPerCta : m * p.ts.i + threadIdx.x] : 0u;
  }
#pragma unroll
  for (int m = 0; m < kMaxRow / 2; ++m) {
    const int e = threadIdx.x + m * kRowsPerCta;
    if (e < R * s) sS[e] = vs[m];
  }
#pragma unroll
  for (int m = 0; m < kMaxRow; ++m) {
    if (t_rows) {
      const int e = threadIdx.x + m * kRowsPerCta;
      if (e < R * n) sT[e] = vt[m];
    } else if (m < n && (int)threadIdx.x < R) {
      sT[threadIdx.x * n + m] = vt[m];
    }
  }
  __syncthreads();
  uint32_t* Xb = p.X + q * p.xs.q + (long long)h0 * w;
  RowWalk x(threadIdx.x, w, p.magic_w);
  for (int e = threadIdx.x; e < R * w; e += kRowsPerCta, x.next())
    Xb[e] = x.i < s ? sS[x.h * s + x.i] : sT[x.h * n + x.i - s];
  for (int j = 0; j < p.k; ++j) {
    const int a = p.w[j].a;
    uint32_t* d = p.cache + p.w[j].offset + q * p.w[j].stride + (long long)h0 * s;
    RowWalk c(threadIdx.x, s, p.magic_s);
    for (int e = threadIdx.x; e < R * s; e += kRowsPerCta, c.next()) {
      const int i = a + c.i;
      d[e] = i < s ? sS[c.h * s + i] : sT[c.h * n + i - s];
    }
  }
}

// The same layouts when every run starts on a 16-byte boundary (the bases,
// the per-sequence strides, the plane stride and the windows' offsets and
// strides multiples of four words): the S and T words of the CTA's channels
// come in as 16-byte loads and are kept in shared memory as they lie (S
// [channel][s], T [channel][n] or [plane][channel]), so staging is a plain
// copy: a thread issues all of its (at most four, as s + n <= 16) 16-byte
// loads before its first store.  Then X and every window are written as
// 16-byte stores, each gathering its four words from shared memory (word c of
// channel h's row is S's word c for c < s, else T's word c - s).  A run's
// last words past a multiple of four go one at a time.
constexpr int kStagePieces = kRowsPerCta * kMaxRow / 4 / kRowsPerCta;  // 16-byte loads a thread

template <bool T_ROWS>
struct StagedRow {
  const uint32_t* sS;
  const uint32_t* sT;
  int s, n;
  __device__ uint32_t operator()(int h, int c) const {
    return c < s ? sS[h * s + c] : (T_ROWS ? sT[h * n + c - s] : sT[(c - s) * kRowsPerCta + h]);
  }
};

template <bool T_ROWS>
__global__ void __launch_bounds__(kRowsPerCta) concat_rows_vec_kernel(ConcatParams p) {
  __shared__ __align__(16) uint32_t sS[kRowsPerCta * (kMaxRow / 2)];
  __shared__ __align__(16) uint32_t sT[kRowsPerCta * kMaxRow];
  const int q = blockIdx.y;
  const int h0 = blockIdx.x * kRowsPerCta;
  const int R = min(kRowsPerCta, p.H - h0);
  const int s = p.s, n = p.n, w = s + n;
  const uint32_t* Sb = p.S + q * p.ss.q + (long long)h0 * s;
  const uint32_t* Tb = p.T + q * p.ts.q + (T_ROWS ? (long long)h0 * n : (long long)h0);
  // 16-byte pieces: S's run, then T's run (rows) or each plane's run (planes)
  const int nS4 = (R * s) >> 2, r4 = R >> 2;
  const int nT4 = T_ROWS ? (R * n) >> 2 : n * r4;
  // plane of T piece g: g / r4 as (g * m4) >> 16, exact since g < 15 r4 and
  // r4 <= 64 (the error g (m4 - 2^16 / r4) / 2^16 < g / 2^16 < 1 / r4)
  const int m4 = r4 > 0 ? (65536 + r4 - 1) / r4 : 0;
  uint4 v[kStagePieces];
#pragma unroll
  for (int m = 0; m < kStagePieces; ++m) {
    const int t = threadIdx.x + m * kRowsPerCta;
    const int g = t - nS4;
    if (t < nS4) {
      v[m] = __ldg(reinterpret_cast<const uint4*>(Sb) + t);
    } else if (g < nT4) {
      if (T_ROWS) {
        v[m] = __ldg(reinterpret_cast<const uint4*>(Tb) + g);
      } else {
        const int j = (g * m4) >> 16;
        v[m] = __ldg(reinterpret_cast<const uint4*>(Tb + j * p.ts.i) + (g - j * r4));
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kStagePieces; ++m) {
    const int t = threadIdx.x + m * kRowsPerCta;
    const int g = t - nS4;
    if (t < nS4) {
      reinterpret_cast<uint4*>(sS)[t] = v[m];
    } else if (g < nT4) {
      if (T_ROWS) {
        reinterpret_cast<uint4*>(sT)[g] = v[m];
      } else {
        const int j = (g * m4) >> 16;
        reinterpret_cast<uint4*>(sT + j * kRowsPerCta)[g - j * r4] = v[m];
      }
    }
  }
  // the words past the last whole piece of each run
  for (int e = 4 * nS4 + (int)threadIdx.x; e < R * s; e += kRowsPerCta) sS[e] = __ldg(Sb + e);
  if (T_ROWS) {
    for (int e = 4 * nT4 + (int)threadIdx.x; e < R * n; e += kRowsPerCta) sT[e] = __ldg(Tb + e);
  } else if (R > 4 * r4) {
    const int rt = R - 4 * r4;
    for (int e = threadIdx.x; e < n * rt; e += kRowsPerCta) {
      const int j = e / rt, h = 4 * r4 + e - j * rt;
      sT[j * kRowsPerCta + h] = __ldg(Tb + j * p.ts.i + h);
    }
  }
  __syncthreads();
  const StagedRow<T_ROWS> row{sS, sT, s, n};
  // X: word e of the run is column e % w of row e / w
  uint32_t* Xb = p.X + q * p.xs.q + (long long)h0 * w;
  const int nX4 = (R * w) >> 2;
  for (int f = threadIdx.x; f < nX4; f += kRowsPerCta) {
    int hh[4], ii[4];
    const int e = 4 * f;
    int h = (e * p.magic_w) >> 16, i = e - h * w;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      hh[u] = h;
      ii[u] = i;
      if (++i == w) {
        i = 0;
        ++h;
      }
    }
    reinterpret_cast<uint4*>(Xb)[f] =
        make_uint4(row(hh[0], ii[0]), row(hh[1], ii[1]), row(hh[2], ii[2]), row(hh[3], ii[3]));
  }
  for (int e = 4 * nX4 + (int)threadIdx.x; e < R * w; e += kRowsPerCta) {
    const int h = (e * p.magic_w) >> 16;
    Xb[e] = row(h, e - h * w);
  }
  // windows: all k share their runs' shape, so a thread walks the rows and
  // columns of its four words once and reads them at every window's start
  const int nW4 = (R * s) >> 2;
  for (int f = threadIdx.x; f < nW4; f += kRowsPerCta) {
    int hh[4], ii[4];
    const int e = 4 * f;
    int h = (e * p.magic_s) >> 16, i = e - h * s;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      hh[u] = h;
      ii[u] = i;
      if (++i == s) {
        i = 0;
        ++h;
      }
    }
    for (int j = 0; j < p.k; ++j) {
      const int a = p.w[j].a;
      uint32_t* d = p.cache + p.w[j].offset + q * p.w[j].stride + (long long)h0 * s;
      reinterpret_cast<uint4*>(d)[f] = make_uint4(row(hh[0], a + ii[0]), row(hh[1], a + ii[1]),
                                                  row(hh[2], a + ii[2]), row(hh[3], a + ii[3]));
    }
  }
  for (int e = 4 * nW4 + (int)threadIdx.x; e < R * s; e += kRowsPerCta) {
    const int h = (e * p.magic_s) >> 16, i = e - h * s;
    for (int j = 0; j < p.k; ++j)
      p.cache[p.w[j].offset + q * p.w[j].stride + (long long)h0 * s + e] = row(h, p.w[j].a + i);
  }
}

// Ordinary path, one snapshot copy: reads the window back from X.  One thread
// per cache word (channel e / s, element a + e % s of its row), so the writes
// are contiguous.
__global__ void __launch_bounds__(256) snapshot_copy_kernel(const uint32_t* X, Strides xs,
                                                            uint32_t* cache, Window w, int s,
                                                            int H) {
  const int q = blockIdx.y;
  const int e = blockIdx.x * 256 + threadIdx.x;
  if (e >= H * s) return;
  const int h = e / s, i = e - h * s;
  cache[w.offset + q * w.stride + e] = X[(w.a + i) * xs.i + h * xs.h + q * xs.q];
}

// Word range [lo, hi) a strided buffer covers, in bytes from address 0.
std::pair<uintptr_t, uintptr_t> span(const void* base, int ni, int H, int Q, const Strides& st) {
  const long long last = (ni - 1) * st.i + (long long)(H - 1) * st.h + (long long)(Q - 1) * st.q;
  const uintptr_t lo = (uintptr_t)base;
  return {lo, lo + (uintptr_t)(last + 1) * 4};
}

bool overlap_any(std::vector<std::pair<uintptr_t, uintptr_t>> r) {
  std::sort(r.begin(), r.end());
  for (size_t i = 1; i < r.size(); ++i)
    if (r[i].first < r[i - 1].second) return true;
  return false;
}

// ---------------------------------------------------------------------------
// Rollback-valid prefix
// ---------------------------------------------------------------------------
// Block row layout (int32): stream, start, n_src, key, pos[0..3], src[0..r).
constexpr int kBlockHead = 8;

__device__ __forceinline__ bool valid_block(const int32_t* blk, int r, int p0,
                                            const int32_t* cell_pos, const uint64_t* cell_seq,
                                            int n_cells) {
  const int stream = blk[0], start = blk[1], n_src = blk[2], key = blk[3];
  if (n_src != r || stream != 0 || start < 0 || (long long)start + r > p0) return false;
  for (int c = 0; c < 4; ++c)
    if (blk[4 + c] != start) return false;
  bool key_found = false;
  for (int i = 0; i < r; ++i) {
    const int c = blk[kBlockHead + i];
    if (c == key) key_found = true;
    if (c < 0 || c >= n_cells) return false;
    if (cell_pos[c] < 0 || cell_seq[c] != 1ull || cell_pos[c] != start + i) return false;
  }
  return key_found;
}

constexpr int kPrefixThreads = 1024;

__global__ void __launch_bounds__(kPrefixThreads)
    rollback_prefix_kernel(const int32_t* blocks, int n_blocks, int r, const int32_t* cell_pos,
                           const uint64_t* cell_seq, int n_cells, int p0, int32_t* out) {
  __shared__ int warp_min[kPrefixThreads / 32];
  int first_bad = n_blocks;
  for (int b = threadIdx.x; b < n_blocks; b += kPrefixThreads) {
    if (b >= first_bad) break;
    if (!valid_block(blocks + (long long)b * (kBlockHead + r), r, p0, cell_pos, cell_seq,
                     n_cells)) {
      first_bad = b;
      break;
    }
  }
  for (int o = 16; o > 0; o >>= 1) first_bad = min(first_bad, __shfl_xor_sync(~0u, first_bad, o));
  if ((threadIdx.x & 31) == 0) warp_min[threadIdx.x >> 5] = first_bad;
  __syncthreads();
  if (threadIdx.x < 32) {
    int m = warp_min[threadIdx.x];
    for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(~0u, m, o));
    if (threadIdx.x == 0) *out = m;
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_concat_snapshots(
    const uint32_t* S, const int64_t* s_strides, const uint32_t* T, const int64_t* t_strides,
    uint32_t* X, const int64_t* x_strides, int32_t s, int32_t n, int32_t H, int32_t Q,
    uint32_t* cache, int64_t cache_words, const mla_snapshot_window_t* windows, int32_t k,
    void* stream, int32_t* fused_out) {
  if (!S || !T || !X || !s_strides || !t_strides || !x_strides || (k > 0 && (!cache || !windows))) {
    set_error("concat/snapshot: a pointer is NULL");
    return MLA_ERR_INVALID_ARG;
  }
  if (s < 1 || n < 1 || s + n > kMaxRow || s > kMaxRow / 2 || H < 1 || Q < 1 || k < 0 ||
      k > kMaxWindows || Q > 65535 || (long long)H * (s + n) > (1LL << 30)) {
    set_error("concat/snapshot: need 1 <= s <= 8, 1 <= n, s + n <= 16, 1 <= Q <= 65535, "
              "1 <= H with H (s + n) <= 2^30, 0 <= k <= 8 (s=%d n=%d H=%d Q=%d k=%d)", s, n, H, Q,
              k);
    return MLA_ERR_INVALID_ARG;
  }
  ConcatParams p;
  p.S = S;
  p.T = T;
  p.X = X;
  p.cache = cache;
  p.ss = {s_strides[0], s_strides[1], s_strides[2]};
  p.ts = {t_strides[0], t_strides[1], t_strides[2]};
  p.xs = {x_strides[0], x_strides[1], x_strides[2]};
  for (const Strides* st : {&p.ss, &p.ts, &p.xs}) {
    if (st->i < 0 || st->h < 0 || st->q < 0) {
      set_error("concat/snapshot: strides must not be negative");
      return MLA_ERR_INVALID_ARG;
    }
  }
  p.s = s;
  p.n = n;
  p.magic_w = div_magic(s + n);
  p.magic_s = div_magic(s);
  p.H = H;
  p.Q = Q;
  p.k = k;
  std::vector<std::pair<uintptr_t, uintptr_t>> dest;
  bool rows_overlap = false;
  for (int j = 0; j < k; ++j) {
    const mla_snapshot_window_t& w = windows[j];
    if (w.window_start < 0 || w.window_start + s > s + n || w.cache_offset < 0 ||
        w.sequence_stride < 0 ||
        w.cache_offset + (int64_t)(Q - 1) * w.sequence_stride + (int64_t)H * s > cache_words) {
      set_error("concat/snapshot: window %d (start %d, offset %lld, stride %lld) is outside the "
                "row or the cache of %lld words", j, w.window_start, (long long)w.cache_offset,
                (long long)w.sequence_stride, (long long)cache_words);
      return MLA_ERR_INVALID_ARG;
    }
    p.w[j] = {w.window_start, w.cache_offset, w.sequence_stride};
    std::vector<std::pair<uintptr_t, uintptr_t>> rows;
    for (int q = 0; q < Q; ++q) {
      const uintptr_t lo = (uintptr_t)(cache + w.cache_offset + (int64_t)q * w.sequence_stride);
      rows.push_back({lo, lo + (uintptr_t)H * s * 4});
    }
    rows_overlap = rows_overlap || overlap_any(rows);
    dest.insert(dest.end(), rows.begin(), rows.end());
  }
  // Algorithm 4: fuse only a group of 2..8 windows whose destinations are
  // pairwise disjoint and lie outside S, T and X
  bool fuse = k >= 2 && !rows_overlap && !overlap_any(dest);
  if (fuse) {
    const std::pair<uintptr_t, uintptr_t> others[3] = {span(S, s, H, Q, p.ss), span(T, n, H, Q, p.ts),
                                                       span(X, s + n, H, Q, p.xs)};
    for (const auto& o : others)
      for (const auto& d : dest)
        if (d.first < o.second && o.first < d.second) fuse = false;
  }
  // The staged kernel serves the contiguous row layouts when X shares no word
  // with S or T (a CTA reads its rows before it writes, not before other CTAs
  // write); other layouts take one thread per row.
  const bool t_rows = p.ts.i == 1 && p.ts.h == n;
  const bool t_planes = p.ts.h == 1 && p.ts.i >= H;
  bool staged = p.ss.i == 1 && p.ss.h == s && p.xs.i == 1 && p.xs.h == s + n &&
                (t_rows || t_planes);
  if (staged) {
    const auto x = span(X, s + n, H, Q, p.xs), a = span(S, s, H, Q, p.ss),
               b = span(T, n, H, Q, p.ts);
    staged = !(x.first < a.second && a.first < x.second) &&
             !(x.first < b.second && b.first < x.second);
  }
  const cudaStream_t st = (cudaStream_t)stream;
  const unsigned grid = (unsigned)(((long long)H * Q + 127) / 128);
  const dim3 grid_rows((unsigned)((H + kRowsPerCta - 1) / kRowsPerCta), (unsigned)Q);
  // 16-byte runs: every base, per-sequence stride and window offset and
  // stride (and the plane stride of T) a multiple of four words
  auto a16 = [](const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; };
  bool vec = staged && a16(S) && a16(T) && a16(X) && p.ss.q % 4 == 0 && p.ts.q % 4 == 0 &&
             p.xs.q % 4 == 0 && (t_rows || p.ts.i % 4 == 0) && (k == 0 || a16(cache));
  for (int j = 0; j < k; ++j) vec = vec && p.w[j].offset % 4 == 0 && p.w[j].stride % 4 == 0;
  auto concat = [&](const ConcatParams& c) {
    if (vec && t_rows)
      concat_rows_vec_kernel<true><<<grid_rows, kRowsPerCta, 0, st>>>(c);
    else if (vec)
      concat_rows_vec_kernel<false><<<grid_rows, kRowsPerCta, 0, st>>>(c);
    else if (staged)
      concat_rows_kernel<<<grid_rows, kRowsPerCta, 0, st>>>(c, t_rows ? 1 : 0);
    else
      concat_snapshots_kernel<<<grid, 128, 0, st>>>(c);
  };
  cudaError_t e;
  if (fuse) {
    KernelTimer kt("concat_snapshots", st);
    concat(p);
    e = cudaGetLastError();
  } else {
    ConcatParams c = p;
    c.k = 0;  // the concatenation alone
    {
      KernelTimer kt("concat", st);
      concat(c);
    }
    e = cudaGetLastError();
    const dim3 grid_copy((unsigned)(((long long)H * s + 255) / 256), (unsigned)Q);
    for (int j = 0; j < k && e == cudaSuccess; ++j) {
      KernelTimer kt("snapshot_copy", st);
      snapshot_copy_kernel<<<grid_copy, 256, 0, st>>>(X, p.xs, cache, p.w[j], s, H);
      e = cudaGetLastError();
    }
  }
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (fused_out) *fused_out = fuse ? 1 : 0;
  return MLA_OK;
}

extern "C" mla_status_t mla_rollback_valid_prefix(const int32_t* blocks, int32_t n_blocks,
                                                  int32_t r, const int32_t* cell_pos,
                                                  const uint64_t* cell_seq, int32_t n_cells,
                                                  int32_t p0, int32_t p1, int32_t seq,
                                                  int32_t n_streams, int32_t* prefix_out,
                                                  void* stream) {
  if (prefix_out == nullptr || n_blocks < 0 || r < 1 || n_cells < 0 ||
      (n_blocks > 0 && blocks == nullptr) || (n_cells > 0 && (!cell_pos || !cell_seq))) {
    set_error("rollback prefix: bad arguments (n_blocks=%d r=%d n_cells=%d)", n_blocks, r,
              n_cells);
    return MLA_ERR_INVALID_ARG;
  }
  // Algorithm 1's global guards: one stream, sequence 0, a removal from a
  // non-negative position to the end; otherwise nothing is retained
  const bool keep = n_streams == 1 && seq == 0 && p0 >= 0 && p1 < 0;
  const cudaStream_t st = (cudaStream_t)stream;
  {
    KernelTimer kt("rollback_prefix", st);
    rollback_prefix_kernel<<<1, kPrefixThreads, 0, st>>>(blocks, keep ? n_blocks : 0, r,
                                                          cell_pos, cell_seq, n_cells, p0,
                                                          prefix_out);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
