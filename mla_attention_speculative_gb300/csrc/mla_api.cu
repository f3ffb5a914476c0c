// C ABI of libmla.so: argument validation, the crossover dispatcher, the
// workspace plan and the launch of the kernels of the chosen branch.
//
// Crossover: "One guard, 110x off the verify step" (sections "The threshold is
// not a constant" and "The change") and the mlx-lm pull request "fix: Speed up
// multi-token decode by computing the absorbed MLA threshold" (opening section
// for the finite-cache form, reviewer comment for exact integer arithmetic).

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "mla_internal.h"

namespace mla {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

// ---------------------------------------------------------------------------
// Crossover threshold, exact integer arithmetic
// ---------------------------------------------------------------------------

// floor(num / den) for num >= 0, den > 0.
static int64_t floor_div(__int128 num, __int128 den) { return (int64_t)(num / den); }

// Per-head costs ("The threshold is not a constant"): absorbed
// 2*L*T*r + L*r*d, materialised T*r*d + L*T*d.  Summed over a batch and
// solved for L: L <= r*d*S / (B*r*d + (2r-d)*S), S = sum of T.  B == 1 is
// the pull request's finite-cache formula; S -> infinity is the helper's
// r*d/(2r-d).  The helper's guards: a non-positive 2r-d gives 1, and the
// answer is never below 1.
static int64_t threshold_sum(int64_t r, int64_t n, int64_t v, int64_t batch, __int128 sumT,
                             bool limit) {
  const int64_t d = n + v;
  const int64_t denom_lim = 2 * r - d;
  if (denom_lim <= 0) return 1;
  int64_t x;
  if (limit) {
    x = floor_div((__int128)r * d, denom_lim);
  } else {
    const __int128 num = (__int128)r * d * sumT;
    const __int128 den = (__int128)batch * r * d + (__int128)denom_lim * sumT;
    x = floor_div(num, den);
  }
  return x < 1 ? 1 : x;
}

}  // namespace mla

using namespace mla;

extern "C" int64_t mla_max_absorbed_queries(int32_t r, int32_t n, int32_t v, int64_t cache_len) {
  if (r <= 0 || n <= 0 || v <= 0) return -1;
  return threshold_sum(r, n, v, 1, cache_len > 0 ? (__int128)cache_len : 0, cache_len <= 0);
}

extern "C" int64_t mla_max_absorbed_queries_batch(int32_t r, int32_t n, int32_t v,
                                                  const int32_t* lens, int32_t batch) {
  if (r <= 0 || n <= 0 || v <= 0 || lens == nullptr || batch < 1) return -1;
  __int128 s = 0;
  for (int32_t b = 0; b < batch; ++b) {
    if (lens[b] < 1) return -1;
    s += lens[b];
  }
  return threshold_sum(r, n, v, batch, s, false);
}

namespace mla {

// ---------------------------------------------------------------------------
// Validation and planning
// ---------------------------------------------------------------------------

static bool geometry_ok(const mla_geometry_t* g) {
  if (g == nullptr) { set_error("geometry is NULL"); return false; }
  if (g->num_heads < 1 || g->kv_lora_rank < 1 || g->qk_nope_dim < 1 || g->v_dim < 1 ||
      g->rope_dim < 0) {
    set_error("geometry has a non-positive dimension (H=%d r=%d n=%d v=%d rope=%d)",
              g->num_heads, g->kv_lora_rank, g->qk_nope_dim, g->v_dim, g->rope_dim);
    return false;
  }
  if (g->dtype != MLA_DTYPE_BF16 && g->dtype != MLA_DTYPE_FP32) {
    set_error("unknown dtype %d", g->dtype);
    return false;
  }
  // every row of every operand is a whole number of 16-byte vectors
  const int eb = g->dtype == MLA_DTYPE_BF16 ? 2 : 4;
  const int dims[4] = {g->kv_lora_rank, g->qk_nope_dim, g->v_dim, g->rope_dim};
  for (int i = 0; i < 4; ++i) {
    if ((dims[i] * eb) % 16 != 0) {
      set_error("dimension %d is not a multiple of %d elements", dims[i], 16 / eb);
      return false;
    }
  }
  if (g->kv_lora_rank > 1024 || g->qk_nope_dim > 512 || g->v_dim > 512 || g->rope_dim > 128) {
    set_error("geometry beyond supported maxima (r<=1024, n<=512, v<=512, rope<=128)");
    return false;
  }
  return true;
}

static bool lens_ok(const int32_t* lens, int32_t batch, int32_t L) {
  if (batch < 1 || batch > 65535) {
    set_error("batch %d outside [1, 65535]", batch);  // (a grid dimension)
    return false;
  }
  if (L < 1) { set_error("L %d < 1", L); return false; }
  if (lens == nullptr) { set_error("cache_lens_host is NULL"); return false; }
  for (int32_t b = 0; b < batch; ++b) {
    if (lens[b] < L) {
      set_error("cache_lens[%d] = %d is smaller than L = %d (T includes the new rows)", b,
                lens[b], L);
      return false;
    }
  }
  return true;
}

static constexpr int kGenericRowsPerCTA = 4; // one warp per query row

// Finish time of one sequence's split-KV clusters on `slots` cluster slots,
// each cluster starting on the slot that frees first, in launch order (piece
// index outermost): (S - 1) x R pieces of c KV tiles, then R pieces of the
// tail, each costing its tiles plus o.  After the full pieces, P - r slots
// are free at q A and r at (q + 1) A (F = q P + r full pieces of cost A); the
// tail pieces go to whichever group frees first, a group's worth at a time.
int64_t pieces_makespan(int64_t R, int64_t klen, int64_t c, int64_t slots, int64_t o) {
  const int64_t S = (klen + c - 1) / c;
  const int64_t A = c + o, Bt = klen - (S - 1) * c + o;
  const int64_t F = (S - 1) * R, q = F / slots, r = F % slots;
  int64_t t1 = q * A, n1 = slots - r, t2 = (q + 1) * A, n2 = r;
  int64_t span = r > 0 ? t2 : t1, left = R;
  while (left > 0) {
    const bool first = n2 == 0 || t1 <= t2;
    int64_t& t = first ? t1 : t2;
    const int64_t n = first ? n1 : n2;
    const int64_t take = left < n ? left : n;
    left -= take;
    span = span > t + Bt ? span : t + Bt;
    t += Bt;
  }
  return span;
}

int device_sm_count() {
  constexpr int kDefault = 152;  // GB300: 2 dies x 76 SMs
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int cached[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return kDefault;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (dev < kMaxDevices && cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    sms = kDefault;
  }
  if (dev < kMaxDevices) cached[dev] = sms;
  return sms;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int choose_branch(const mla_geometry_t* g, int32_t L, const int32_t* lens, int32_t batch,
                         int32_t mode) {
  if (mode == MLA_MODE_ABSORBED) return MLA_BRANCH_ABSORBED;
  if (mode == MLA_MODE_MATERIALISED) return MLA_BRANCH_MATERIALISED;
  const int64_t thr =
      mla_max_absorbed_queries_batch(g->kv_lora_rank, g->qk_nope_dim, g->v_dim, lens, batch);
  return L <= thr ? MLA_BRANCH_ABSORBED : MLA_BRANCH_MATERIALISED;
}

static mla_status_t make_plan(const mla_geometry_t* g, int32_t batch, int32_t L,
                              const int32_t* lens, int32_t mode, Plan* p) {
  if (!geometry_ok(g) || !lens_ok(lens, batch, L)) return MLA_ERR_INVALID_ARG;
  if (mode != MLA_MODE_AUTO && mode != MLA_MODE_ABSORBED && mode != MLA_MODE_MATERIALISED) {
    set_error("unknown mode %d", mode);
    return MLA_ERR_INVALID_ARG;
  }
  p->B = batch;
  p->L = L;
  p->H = g->num_heads;
  p->r = g->kv_lora_rank;
  p->n = g->qk_nope_dim;
  p->v = g->v_dim;
  p->rope = g->rope_dim;
  p->dtype = g->dtype;
  p->scale = g->softmax_scale > 0.f ? g->softmax_scale
                                    : (float)(1.0 / std::sqrt((double)(p->n + p->rope)));
  p->branch = choose_branch(g, L, lens, batch, mode);
  p->Tmax = 0;
  p->sumT = 0;
  for (int b = 0; b < batch; ++b) {
    p->Tmax = lens[b] > p->Tmax ? lens[b] : p->Tmax;
    p->sumT += lens[b];
  }

  // Generic split-KV: enough CTAs (one per 4 query rows per piece) to cover
  // the GPU a few times over, pieces a multiple of 64 rows.
  const int64_t rows = (int64_t)L * p->H;
  const size_t eb = p->dtype == MLA_DTYPE_BF16 ? 2 : 4;
  const int64_t num_sms = device_sm_count();
  const size_t nrow = (size_t)batch * rows;
  {
    SplitPlan& g = p->generic;
    const int64_t row_ctas =
        (int64_t)batch * ((rows + kGenericRowsPerCTA - 1) / kGenericRowsPerCTA);
    const int64_t want = 4 * num_sms;
    int64_t splits = (want + row_ctas - 1) / row_ctas;
    const int64_t max_splits = (p->Tmax + 63) / 64;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t chunk = (p->Tmax + splits - 1) / splits;
    chunk = (chunk + 63) / 64 * 64;
    g.chunk = (int)chunk;
    g.splits = (int)((p->Tmax + chunk - 1) / chunk);
    const int dv = p->branch == MLA_BRANCH_ABSORBED ? p->r : p->v;
    size_t off = 0;
    if (p->branch == MLA_BRANCH_ABSORBED) {
      g.off_qlat = off;
      off = align256(off + nrow * p->r * sizeof(float));
    } else {
      g.off_exp = off;
      off = align256(off + (size_t)batch * p->Tmax * p->H * (p->n + p->v) * eb);
    }
    g.off_opart = off;
    off = align256(off + nrow * g.splits * dv * sizeof(float));
    g.off_ml = off;
    off = align256(off + nrow * g.splits * 2 * sizeof(float));
    g.bytes = off;
  }
  p->fast_ok = p->branch == MLA_BRANCH_ABSORBED ? fast_absorbed_supported(*p)
                                                : fast_materialised_supported(*p);
  if (p->fast_ok && p->branch == MLA_BRANCH_MATERIALISED) {
    // no split-KV: one CTA per (128-row query tile, head, sequence) walks the
    // whole visible cache
    SplitPlan& f = p->fast;
    f.chunk = p->Tmax;
    f.splits = 1;
    f.off_exp = 0;
    f.bytes = align256(fast_materialised_workspace(*p));
  } else if (p->fast_ok) {
    // Tensor-core split-KV: clusters of 2 CTAs, one per (128-row tile, piece).
    // Pick the piece length ct (in 64-row KV tiles) that minimises
    // waves x (ct + overhead) over the SMs' cluster slots, where the fixed
    // cost of a cluster (Q load, pipeline fill, writing 128 x 512 fp32
    // partials that the merge reads back) is worth about kClusterOverhead KV
    // tiles; ties go to longer pieces (fewer partials).
    constexpr int64_t kClusterOverhead = 4;
    SplitPlan& f = p->fast;
    const int64_t row_tiles = (rows + 127) / 128;
    const int64_t slots = absorbed_cluster_slots();
    const int64_t max_tiles = (p->Tmax + 63) / 64;
    int64_t ct = max_tiles, best_cost = -1;
    for (int64_t c = max_tiles; c >= 1; --c) {
      int64_t clusters = 0;
      for (int b = 0; b < batch; ++b) clusters += row_tiles * (((lens[b] + 63) / 64 + c - 1) / c);
      const int64_t cost = ((clusters + slots - 1) / slots) * (c + kClusterOverhead);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        ct = c;
      }
    }
    // One sequence whose pieces fit one wave: the clusters launch piece index
    // outermost, so every row tile's short last piece comes last and can run
    // in the gaps the full pieces leave.  Score a few shorter pieces by that
    // list schedule; keep at most 64 pieces, which the fused merge takes.
    // (Plans of several waves keep the wave model: the schedule below is too
    // coarse for them.)
    const int64_t klen0 = (lens[0] + 63) / 64;
    if (batch == 1 && row_tiles * ((klen0 + ct - 1) / ct) <= slots) {
      const int64_t klen = klen0;
      int64_t best_c = ct;
      int64_t best_span = pieces_makespan(row_tiles, klen, ct, slots, kClusterOverhead);
      for (int64_t c = ct - 1; c >= 1 && c >= ct - 8; --c) {
        if ((klen + c - 1) / c > 64) break;
        const int64_t span = pieces_makespan(row_tiles, klen, c, slots, kClusterOverhead);
        if (span < best_span) {
          best_span = span;
          best_c = c;
        }
      }
      // A length that divides the cache evenly leaves no short last piece:
      // every cluster ends together, which the schedule above (a flat
      // overhead per piece) under-rates by about a tile or two.  Take the
      // best such length at or above the choice when it scores within two
      // (no more pieces than the choice, so still one wave).
      int64_t even_c = 0, even_span = 0;
      for (int64_t c = best_c; c <= klen; ++c) {
        if (klen % c != 0) continue;
        const int64_t span = pieces_makespan(row_tiles, klen, c, slots, kClusterOverhead);
        if (span <= best_span + 2 && (even_c == 0 || span < even_span)) {
          even_span = span;
          even_c = c;
        }
      }
      ct = even_c > 0 ? even_c : best_c;
    }
    f.chunk = (int)(ct * 64);
    f.splits = (int)((p->Tmax + f.chunk - 1) / f.chunk);
    size_t off = 0;
    f.off_qlat = off;  // Q tiles: every sequence's rows padded to 128-row tiles
    off = align256(off + (size_t)batch * row_tiles * 128 * p->r * 2);
    f.off_opart = off;  // bf16 O / l of every piece
    off = align256(off + nrow * f.splits * p->r * 2);
    f.off_ml = off;
    off = align256(off + nrow * f.splits * 2 * sizeof(float));
    f.off_olat = off;
    off = align256(off + nrow * p->r * 2);
    f.bytes = off;
  }
  p->ws_bytes = p->fast_ok && p->fast.bytes > p->generic.bytes ? p->fast.bytes : p->generic.bytes;
  p->use(p->generic);
  return MLA_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Every page a position t < T_b needs is in [0, num_pages), and the table is
// wide enough for the longest sequence.
static mla_status_t check_page_table(const int32_t* table, int32_t batch, int32_t max_pages,
                                     const int32_t* lens, int32_t page_size, int32_t num_pages) {
  if (table == nullptr || lens == nullptr || batch < 1 || max_pages < 1 || page_size < 1 ||
      num_pages < 1) {
    set_error("page table check needs a table, lengths, batch, max_pages, page_size and "
              "num_pages >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  for (int32_t b = 0; b < batch; ++b) {
    if (lens[b] < 0) {
      set_error("cache_lens[%d] = %d is negative", b, lens[b]);
      return MLA_ERR_INVALID_ARG;
    }
    const int64_t need = ((int64_t)lens[b] + page_size - 1) / page_size;
    if (need > max_pages) {
      set_error("sequence %d needs %lld pages but the table holds %d per sequence", b,
                (long long)need, max_pages);
      return MLA_ERR_INVALID_ARG;
    }
    for (int64_t j = 0; j < need; ++j) {
      const int32_t id = table[(int64_t)b * max_pages + j];
      if (id < 0 || id >= num_pages) {
        set_error("page_table[%d][%lld] = %d is outside [0, %d)", b, (long long)j, id,
                  num_pages);
        return MLA_ERR_INVALID_ARG;
      }
    }
  }
  return MLA_OK;
}

// MLA_DEBUG_CHECKS=1 in the environment: each call copies the device cache
// lengths (and page table) back to the host and checks them before launching.
static bool debug_checks() {
  static const bool on = [] {
    const char* e = std::getenv("MLA_DEBUG_CHECKS");
    return e != nullptr && e[0] != '\0' && e[0] != '0';
  }();
  return on;
}

static mla_status_t debug_check_device_args(const int32_t* lens_dev, const int32_t* lens_host,
                                            int32_t batch, const int32_t* page_table,
                                            int32_t max_pages, int32_t page_size,
                                            int32_t num_pages, cudaStream_t stream) {
  std::vector<int32_t> lens(batch);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess)
    e = cudaMemcpy(lens.data(), lens_dev, sizeof(int32_t) * batch, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_error("debug check could not read cache_lens_dev: %s", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  for (int32_t b = 0; b < batch; ++b) {
    if (lens[b] != lens_host[b]) {
      set_error("cache_lens_dev[%d] = %d but cache_lens_host[%d] = %d", b, lens[b], b,
                lens_host[b]);
      return MLA_ERR_INVALID_ARG;
    }
  }
  if (page_table == nullptr) return MLA_OK;
  std::vector<int32_t> table((size_t)batch * max_pages);
  e = cudaMemcpy(table.data(), page_table, sizeof(int32_t) * table.size(),
                 cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_error("debug check could not read page_table: %s", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return check_page_table(table.data(), batch, max_pages, lens_host, page_size, num_pages);
}

}  // namespace mla

extern "C" mla_status_t mla_check_page_table(const int32_t* page_table_host, int32_t batch,
                                             int32_t max_pages_per_seq,
                                             const int32_t* cache_lens_host, int32_t page_size,
                                             int32_t num_pages) {
  return check_page_table(page_table_host, batch, max_pages_per_seq, cache_lens_host, page_size,
                          num_pages);
}


extern "C" mla_status_t mla_select_branch(const mla_geometry_t* g, int32_t L,
                                          const int32_t* lens, int32_t batch, int32_t mode,
                                          int32_t* branch) {
  if (branch == nullptr) { set_error("branch output is NULL"); return MLA_ERR_INVALID_ARG; }
  Plan p;
  const mla_status_t st = make_plan(g, batch, L, lens, mode, &p);
  if (st != MLA_OK) return st;
  *branch = p.branch;
  return MLA_OK;
}

extern "C" mla_status_t mla_workspace_bytes(const mla_geometry_t* g, int32_t batch, int32_t L,
                                            const int32_t* lens, int32_t mode, size_t* bytes) {
  if (bytes == nullptr) { set_error("bytes output is NULL"); return MLA_ERR_INVALID_ARG; }
  Plan p;
  const mla_status_t st = make_plan(g, batch, L, lens, mode, &p);
  if (st != MLA_OK) return st;
  *bytes = p.ws_bytes;
  return MLA_OK;
}

namespace mla {

// The plan of a sparse (top-k) call: the absorbed branch, with the pieces
// cut along each row's index list of topk_len entries instead of [0, T_b).
static mla_status_t make_sparse_plan(const mla_geometry_t* g, int32_t batch, int32_t L,
                                     const int32_t* lens_host, int32_t topk_len, Plan* p) {
  if (!geometry_ok(g) || !lens_ok(lens_host, batch, L)) return MLA_ERR_INVALID_ARG;
  if (topk_len < 1) {
    set_error("topk_len %d < 1", topk_len);
    return MLA_ERR_INVALID_ARG;
  }
  // the planner sizes pieces from these lengths (at least L, which it requires)
  std::vector<int32_t> plan_lens(batch, topk_len > L ? topk_len : L);
  const mla_status_t st = make_plan(g, batch, L, plan_lens.data(), MLA_MODE_ABSORBED, p);
  if (st != MLA_OK) return st;
  // the tensor-core kernel takes one verify row per 128-row tile
  if (p->fast_ok && p->H % 128 != 0) {
    p->fast_ok = false;
    p->ws_bytes = p->generic.bytes;
  }
  return MLA_OK;
}

// Validation and launch shared by the dense and the sparse entry points
// (topk == NULL: dense).
static mla_status_t verify_impl(
    const mla_geometry_t* g, const void* q_nope, const void* q_rope, const void* c_kv,
    const void* k_rope, int64_t c_kv_row_stride, int64_t k_rope_row_stride,
    int64_t seq_stride_rows, const void* W_UK, const void* W_UV, const int32_t* lens_dev,
    const int32_t* lens_host, int32_t batch, int32_t L, const int32_t* topk, int32_t topk_len,
    const int32_t* page_table, int32_t page_size, int32_t max_pages_per_seq, int32_t num_pages,
    int32_t mode, void* out, void* workspace, size_t workspace_bytes, void* stream,
    int32_t* branch_taken) {
  Plan p;
  mla_status_t st = topk ? make_sparse_plan(g, batch, L, lens_host, topk_len, &p)
                         : make_plan(g, batch, L, lens_host, mode, &p);
  if (st != MLA_OK) return st;
  if (topk) {
    // the real cache lengths bound the addresses the list may name
    p.Tmax = 0;
    for (int b = 0; b < batch; ++b) p.Tmax = lens_host[b] > p.Tmax ? lens_host[b] : p.Tmax;
    if (!aligned16(topk)) {
      set_error("topk is not 16-byte aligned");
      return MLA_ERR_INVALID_ARG;
    }
  }

  const void* ptrs[] = {q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, lens_dev, out};
  const char* names[] = {"q_nope", "q_rope", "c_kv", "k_rope", "W_UK", "W_UV",
                         "cache_lens_dev", "out"};
  for (int i = 0; i < 8; ++i) {
    if (ptrs[i] == nullptr) { set_error("%s is NULL", names[i]); return MLA_ERR_INVALID_ARG; }
    if (!aligned16(ptrs[i])) {
      set_error("%s is not 16-byte aligned", names[i]);
      return MLA_ERR_INVALID_ARG;
    }
  }
  const int64_t eb = p.dtype == MLA_DTYPE_BF16 ? 2 : 4;
  if (c_kv_row_stride < p.r || k_rope_row_stride < p.rope || (c_kv_row_stride * eb) % 16 ||
      (k_rope_row_stride * eb) % 16) {
    set_error("row strides (%lld, %lld) must cover r/rope and be 16-byte multiples",
              (long long)c_kv_row_stride, (long long)k_rope_row_stride);
    return MLA_ERR_INVALID_ARG;
  }
  if (page_table == nullptr) {
    if (seq_stride_rows < p.Tmax && batch > 1) {
      set_error("seq_stride_rows %lld < longest cache %d", (long long)seq_stride_rows, p.Tmax);
      return MLA_ERR_INVALID_ARG;
    }
  } else {
    if (page_size < 1 || max_pages_per_seq < 1 || num_pages < 1) {
      set_error("paged cache needs page_size, max_pages_per_seq, num_pages >= 1");
      return MLA_ERR_INVALID_ARG;
    }
    if ((int64_t)max_pages_per_seq * page_size < p.Tmax) {
      set_error("page table of %d pages x %d rows cannot hold %d positions", max_pages_per_seq,
                page_size, p.Tmax);
      return MLA_ERR_INVALID_ARG;
    }
    if (!aligned16(page_table)) {
      set_error("page_table is not 16-byte aligned");
      return MLA_ERR_INVALID_ARG;
    }
  }
  if (workspace_bytes < p.ws_bytes || (p.ws_bytes > 0 && workspace == nullptr)) {
    set_error("workspace of %zu bytes is smaller than the %zu this call needs",
              workspace_bytes, p.ws_bytes);
    return MLA_ERR_WORKSPACE;
  }
  if (workspace != nullptr && ((uintptr_t)workspace & 255u)) {
    set_error("workspace is not 256-byte aligned");
    return MLA_ERR_INVALID_ARG;
  }

  if (debug_checks()) {
    st = debug_check_device_args(lens_dev, lens_host, batch, page_table, max_pages_per_seq,
                                 page_size, num_pages, (cudaStream_t)stream);
    if (st != MLA_OK) return st;
  }

  Args a;
  a.q_nope = q_nope;
  a.q_rope = q_rope;
  a.cache.c_kv = c_kv;
  a.cache.k_rope = k_rope;
  a.cache.ckv_stride = c_kv_row_stride;
  a.cache.kr_stride = k_rope_row_stride;
  a.cache.seq_stride = seq_stride_rows;
  a.cache.page_table = page_table;
  a.cache.page_size = page_size;
  a.cache.max_pages = max_pages_per_seq;
  a.cache.num_pages = num_pages;
  a.W_UK = W_UK;
  a.W_UV = W_UV;
  a.lens = lens_dev;
  a.topk = topk;
  a.topk_k = topk ? topk_len : 0;
  a.out = out;
  a.ws = (char*)workspace;
  a.stream = (cudaStream_t)stream;

  // The tensor-core kernels address the cache with 32-bit TMA row
  // coordinates and read 64-row boxes that must not straddle pages.
  const int64_t cache_rows = page_table ? (int64_t)num_pages * page_size
                                        : (int64_t)(batch - 1) * seq_stride_rows + p.Tmax;
  const bool fast = p.fast_ok && (page_table == nullptr || page_size % 64 == 0) &&
                    cache_rows < ((int64_t)1 << 31);
  // (the generic kernels' split plan was made with the list length as T too)
  cudaError_t e;
  if (fast) {
    p.use(p.fast);
    e = p.branch == MLA_BRANCH_ABSORBED ? launch_fast_absorbed(p, a)
                                        : launch_fast_materialised(p, a);
  } else {
    e = p.branch == MLA_BRANCH_ABSORBED ? launch_generic_absorbed(p, a)
                                        : launch_generic_materialised(p, a);
  }
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (branch_taken) *branch_taken = p.branch;
  return MLA_OK;
}

}  // namespace mla

extern "C" mla_status_t mla_verify_attention(
    const mla_geometry_t* g, const void* q_nope, const void* q_rope, const void* c_kv,
    const void* k_rope, int64_t c_kv_row_stride, int64_t k_rope_row_stride,
    int64_t seq_stride_rows, const void* W_UK, const void* W_UV, const int32_t* lens_dev,
    const int32_t* lens_host, int32_t batch, int32_t L, const int32_t* page_table,
    int32_t page_size, int32_t max_pages_per_seq, int32_t num_pages, int32_t mode, void* out,
    void* workspace, size_t workspace_bytes, void* stream, int32_t* branch_taken) {
  return verify_impl(g, q_nope, q_rope, c_kv, k_rope, c_kv_row_stride, k_rope_row_stride,
                     seq_stride_rows, W_UK, W_UV, lens_dev, lens_host, batch, L, nullptr, 0,
                     page_table, page_size, max_pages_per_seq, num_pages, mode, out, workspace,
                     workspace_bytes, stream, branch_taken);
}

extern "C" mla_status_t mla_sparse_workspace_bytes(const mla_geometry_t* g, int32_t batch,
                                                   int32_t L, const int32_t* lens_host,
                                                   int32_t topk_len, size_t* bytes) {
  if (bytes == nullptr) { set_error("bytes output is NULL"); return MLA_ERR_INVALID_ARG; }
  Plan p;
  const mla_status_t st = make_sparse_plan(g, batch, L, lens_host, topk_len, &p);
  if (st != MLA_OK) return st;
  *bytes = p.ws_bytes;
  return MLA_OK;
}

extern "C" mla_status_t mla_verify_attention_sparse(
    const mla_geometry_t* g, const void* q_nope, const void* q_rope, const void* c_kv,
    const void* k_rope, int64_t c_kv_row_stride, int64_t k_rope_row_stride,
    int64_t seq_stride_rows, const void* W_UK, const void* W_UV, const int32_t* lens_dev,
    const int32_t* lens_host, int32_t batch, int32_t L, const int32_t* topk, int32_t topk_len,
    const int32_t* page_table, int32_t page_size, int32_t max_pages_per_seq, int32_t num_pages,
    void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (topk == nullptr) {
    set_error("topk is NULL");
    return MLA_ERR_INVALID_ARG;
  }
  return verify_impl(g, q_nope, q_rope, c_kv, k_rope, c_kv_row_stride, k_rope_row_stride,
                     seq_stride_rows, W_UK, W_UV, lens_dev, lens_host, batch, L, topk, topk_len,
                     page_table, page_size, max_pages_per_seq, num_pages, MLA_MODE_ABSORBED, out,
                     workspace, workspace_bytes, stream, nullptr);
}

extern "C" const char* mla_status_string(int32_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    default: return "MLA_ERR_UNKNOWN";
  }
}

extern "C" const char* mla_last_error(void) { return g_err; }

extern "C" mla_status_t mla_device_status(int32_t* code, int32_t clear) {
  const int words[5] = {absorbed_device_status(clear != 0), materialised_device_status(clear != 0),
                        generic_device_status(clear != 0), selftest_device_status(clear != 0),
                        indexer_device_status(clear != 0)};
  int v = 0;
  for (int w : words) {
    if (w < 0) {
      v = -1;
      break;
    }
    if (v == 0) v = w;
  }
  if (code) *code = v;
  if (v < 0) {
    set_error("could not read the device status word");
    return MLA_ERR_CUDA;
  }
  if (v >= kBadPageSite) {
    set_error("a kernel met a page id outside [0, num_pages) (site %d); the positions of that "
              "page read as zeros",
              v);
    return MLA_ERR_INVALID_ARG;
  }
  if (v != 0) {
    set_error("a bounded device wait ran out (site %d)", v);
    return MLA_ERR_TIMEOUT;
  }
  return MLA_OK;
}

extern "C" mla_status_t mla_selftest_bounded_wait(void* stream) {
  const cudaError_t e = launch_wait_selftest((cudaStream_t)stream);
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

extern "C" int32_t mla_version(void) { return 100; }
