// zr_plan.cpp — host planner (see zr_plan.h).
//
// Broadcast rule: Zero book, Operator page, section 广播 — compare from the
// last dim; equal, or one side 1, or one side missing.  A size-1 input dim
// reads coordinate 0, which is a stride of 0 here, so no broadcast operand is
// ever materialised.  Strides: Tensor page, section 形状与步长.
#include "zr_plan.h"

#include <algorithm>
#include <cstdio>
#include <limits>

namespace zr {

namespace {

constexpr int64_t kI64Max = std::numeric_limits<int64_t>::max();

bool mul_overflows(int64_t a, int64_t b) { return a != 0 && b > kI64Max / a; }

uint32_t pow2_ceil(uint64_t v) {
  uint32_t p = 1;
  while (p < v && p < (1u << 31)) p *= 2;
  return p;
}
uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

// Target elements per CTA: enough CTAs to fill 152 SMs several times over,
// and enough bytes per thread to keep loads in flight.
uint64_t elems_per_cta_target(uint64_t total) {
  uint64_t e = total / 1216;
  if (e < 4096) e = 4096;
  if (e > 32768) e = 32768;
  return e;
}

// Column lanes for a row of nvcol vectors: a power of two <= 256 with the
// least padding, preferring wider.
uint32_t pick_tx(uint64_t nvcol) {
  if (nvcol <= 32) return pow2_ceil(nvcol);
  uint32_t best = 32;
  uint64_t best_waste = ceil_div(nvcol, 32) * 32 - nvcol;
  for (uint32_t tx = 64; tx <= 256; tx *= 2) {
    const uint64_t waste = ceil_div(nvcol, tx) * tx - nvcol;
    if (waste <= best_waste) { best = tx; best_waste = waste; }
  }
  return best;
}

// Fill of the last wave when `ctas` CTAs run `wave` at a time (1 for a whole
// number of waves).  Grids of 6 waves or more count as full: their CTAs start
// staggered, and resizing their tiles measured no gain.
constexpr uint64_t kFullWaves = 6;
double wave_fill(uint64_t ctas, uint64_t wave) {
  if (ctas == 0) return 0.0;
  const uint64_t waves = ceil_div(ctas, wave);
  if (waves >= kFullWaves) return 1.0;
  return double(ctas) / double(waves * wave);
}

// Block count n along one split of a grid with F CTAs per block of that
// split, within [lo, hi]: either pref, or for k whole waves around pref's,
// the most blocks that fit in k waves, whichever fills its last wave best
// (pref on ties).  real(n) is the count the tile size implied by n really
// gives (tile sizes are rounded).
template <class Real>
uint64_t fit_waves(uint64_t pref, uint64_t lo, uint64_t hi, uint64_t F, uint64_t wave, Real real) {
  uint64_t pick = pref;
  double best = wave_fill(F * real(pref), wave);
  const uint64_t k0 = ceil_div(F * real(pref), wave);
  if (k0 >= kFullWaves || best >= 1.0) return pick;
  for (uint64_t k = k0 > 2 ? k0 - 2 : 1; k <= k0 + 1; ++k) {
    uint64_t n = k * wave / F;
    n = std::min(std::max(n, lo), hi);
    if (n == 0) continue;
    const double f = wave_fill(F * real(n), wave);
    if (f > best + 1e-9) { best = f; pick = n; }
  }
  return pick;
}

// Flat elementwise plans: items per load batch of the kernel (4 in flight per
// thread x 256 threads), and the largest item count (item indices and the
// batch loop stay within 32 bits).
constexpr uint64_t kFlatBatch = 4 * kThreads;
constexpr uint64_t kFlatMaxItems = (uint64_t(1) << 32) - (uint64_t(1) << 20);

// Thread layout of the combine pass: jx outputs x sy slot lanes (powers of
// two, jx * sy <= 256).  Few slots: one output per thread, summed serially
// (no tree).  Many slots: rows of jx consecutive outputs (32, or down to 8 =
// one 32-byte sector, until there are about two CTAs per SM) and the lanes
// left over go to the slots, so each thread has few partials to load.
void combine_layout(CombinePlan* c) {
  if (c->vec == 0) c->vec = 1;
  const uint64_t units = ceil_div(c->nout, c->vec);  // output groups
  uint32_t jx;
  if (c->nslots <= 16) {
    jx = kThreads;
  } else if (units < 8) {
    jx = pow2_ceil(units);
  } else {
    jx = 32;
    while (jx > 8 && ceil_div(units, jx) < 2 * 152) jx /= 2;
  }
  if (jx > kThreads) jx = kThreads;
  const uint32_t sy_max = kThreads / jx;
  c->jx = jx;
  c->sy = std::min<uint32_t>(sy_max, pow2_ceil(c->nslots));
}

void fill_decomp(Decomp* dc, const Prob& P, const int* dims, int nd) {
  // dims: outer dims in row-major order; the decomposition is innermost first.
  dc->n = nd;
  for (int i = 0; i < nd; ++i) {
    const int d = dims[nd - 1 - i];
    dc->div[i] = make_fastdiv(static_cast<uint32_t>(P.size[d]));
    for (int k = 0; k < kMaxOperands; ++k) dc->stride[k][i] = P.st[k][d];
  }
  for (int i = nd; i < kMaxDims; ++i) {
    dc->div[i] = make_fastdiv(1);
    for (int k = 0; k < kMaxOperands; ++k) dc->stride[k][i] = 0;
  }
}

// VEC = V is allowed when the inner dim is a multiple of V and every slot
// that is read or written with unit inner stride starts aligned to V elements
// and every row start stays aligned.
bool vec_ok(const Prob& P, int V, uint32_t slots, const void* const* ptrs) {
  const int n = P.n;
  if (P.size[n - 1] % V != 0) return false;
  bool any_unit = false;
  for (int k = 0; k < kMaxOperands; ++k) {
    if (!(slots & (1u << k))) continue;
    if (P.st[k][n - 1] != 1) continue;
    any_unit = true;
    if (reinterpret_cast<uintptr_t>(ptrs[k]) % uintptr_t(V * P.es) != 0) return false;
    for (int d = 0; d < n - 1; ++d)
      if (P.st[k][d] % V != 0) return false;
  }
  return any_unit;
}

// Elements per vector access: 16 bytes where alignment allows (4 floats or
// 8 bfloat16), for bfloat16 else 8 bytes (4 elements), else one element.
// extra: another pointer that must share the alignment (or null).
int pick_vec(const Prob& P, uint32_t slots, const void* const* ptrs, const void* extra) {
  const int cands[2] = {P.es == 2 ? 8 : 4, 4};
  for (int i = 0; i < (P.es == 2 ? 2 : 1); ++i) {
    const int V = cands[i];
    if (vec_ok(P, V, slots, ptrs) &&
        (!extra || reinterpret_cast<uintptr_t>(extra) % uintptr_t(V * P.es) == 0))
      return V;
  }
  return 1;
}

}  // namespace

uint64_t red_smem_bytes(const RedPlan& p, int vec, uint32_t stages, uint32_t stage_ns) {
  const uint64_t table_rows = std::min<uint64_t>(p.rows_per_blk, kMaxTileRows);
  const uint64_t red_floats = p.inner_kept ? uint64_t(kThreads) * vec : uint64_t(kThreads);
  return table_rows * kMaxOperands * sizeof(int64_t) +
         std::max<uint64_t>(red_floats * sizeof(float), uint64_t(stages) * stage_ns * kStageBatchBytes);
}

void combine_vectorize(CombinePlan* c) {
  c->vec = 1;
  if (c->nout % 4 == 0 && c->nout >= 64 * 152 && reinterpret_cast<uintptr_t>(c->partial) % 16 == 0)
    c->vec = 4;
  combine_layout(c);
}

uint64_t combine_blocks(const CombinePlan& c) {
  return ceil_div(ceil_div(c.nout, c.vec ? c.vec : 1), c.jx);
}

int read_tensor(const zr_tensor& t, TDesc* d) {
  if (t.ndim < 0 || t.ndim > kMaxDims) return ZR_ERR_RANK;
  if (t.ndim > 0 && t.sizes == nullptr) return ZR_ERR_NULL;
  d->ptr = static_cast<const float*>(t.data);
  d->nd = t.ndim;
  int64_t n = 1;
  for (int i = 0; i < t.ndim; ++i) {
    const int64_t s = t.sizes[i];
    if (s < 0) return ZR_ERR_SIZE;
    if (mul_overflows(n, s) && s != 0) return ZR_ERR_SIZE;
    d->size[i] = s;
    n *= s;
  }
  d->numel = n;
  if (t.strides) {
    for (int i = 0; i < t.ndim; ++i) {
      if (t.strides[i] < 0) return ZR_ERR_SIZE;
      d->stride[i] = t.strides[i];
    }
  } else {
    contiguous_strides(t.ndim, d->size, d->stride);
  }
  d->extent = 0;
  if (n > 0) {
    int64_t e = 0;
    for (int i = 0; i < t.ndim; ++i) {
      if (mul_overflows(d->size[i] - 1, d->stride[i])) return ZR_ERR_SIZE;
      const int64_t span = (d->size[i] - 1) * d->stride[i];
      if (e > kI64Max - span) return ZR_ERR_SIZE;
      e += span;
    }
    if (e > kI64Max / 4 - 1) return ZR_ERR_SIZE;
    d->extent = e + 1;
  }
  return ZR_OK;
}

void contiguous_strides(int nd, const int64_t* size, int64_t* stride) {
  int64_t s = 1;
  for (int i = nd - 1; i >= 0; --i) {
    stride[i] = s;
    s *= size[i] > 0 ? size[i] : 1;
  }
}

int broadcast_sizes(int nda, const int64_t* sa, int ndb, const int64_t* sb, int* nd,
                    int64_t* so) {
  if (nda < 0 || nda > kMaxDims || ndb < 0 || ndb > kMaxDims) return ZR_ERR_RANK;
  const int n = nda > ndb ? nda : ndb;
  for (int k = 0; k < n; ++k) {
    const int64_t x = k < nda ? sa[nda - 1 - k] : 1;
    const int64_t y = k < ndb ? sb[ndb - 1 - k] : 1;
    if (x < 0 || y < 0) return ZR_ERR_SIZE;
    int64_t o;
    if (x == y) o = x;
    else if (x == 1) o = y;
    else if (y == 1) o = x;
    else return ZR_ERR_SHAPE;
    so[n - 1 - k] = o;
  }
  *nd = n;
  return ZR_OK;
}

void align_strides(const TDesc& x, int n, const int64_t* out_size, int64_t* st) {
  for (int od = 0; od < n; ++od) {
    const int d = od - (n - x.nd);
    st[od] = (d < 0 || x.size[d] == 1 || out_size[od] == 1) ? 0 : x.stride[d];
  }
}

void grad_index_strides(const TDesc& x, int n, const int64_t* out_size, int64_t* st) {
  int64_t cs[kMaxDims];
  contiguous_strides(x.nd, x.size, cs);
  for (int od = 0; od < n; ++od) {
    const int d = od - (n - x.nd);
    st[od] = (d < 0 || x.size[d] == 1 || out_size[od] == 1) ? 0 : cs[d];
  }
}

int coalesce(int n, const int64_t* size, const int64_t (*st)[kMaxDims], uint32_t active,
             int order_slot, Prob* P) {
  int dims[kMaxDims];
  int nd = 0;
  for (int d = 0; d < n; ++d)
    if (size[d] != 1) dims[nd++] = d;
  if (order_slot >= 0) {
    std::stable_sort(dims, dims + nd, [&](int x, int y) {
      return st[order_slot][x] > st[order_slot][y];
    });
  }
  // Merge from the innermost dim outwards: dim d folds into the current
  // outermost merged dim c when every active slot has st[d] == st[c] * size[c].
  int64_t msize[kMaxDims];
  int64_t mst[kProbSlots][kMaxDims];
  int m = 0;  // merged dims stored innermost first
  for (int i = nd - 1; i >= 0; --i) {
    const int d = dims[i];
    bool merge = m > 0;
    if (merge) {
      for (int k = 0; k < kProbSlots && merge; ++k) {
        if (!(active & (1u << k))) continue;
        if (mul_overflows(mst[k][m - 1], msize[m - 1])) merge = false;
        else if (st[k][d] != mst[k][m - 1] * msize[m - 1]) merge = false;
      }
    }
    if (merge) {
      msize[m - 1] *= size[d];
    } else {
      msize[m] = size[d];
      for (int k = 0; k < kProbSlots; ++k) mst[k][m] = (active & (1u << k)) ? st[k][d] : 0;
      ++m;
    }
  }
  if (m == 0) {  // every dim is 1: one element
    msize[0] = 1;
    for (int k = 0; k < kProbSlots; ++k) mst[k][0] = 0;
    m = 1;
  }
  // An innermost dim of 2^31 or more elements is split into [size / W, W]
  // with W a power of two, so that column indices fit 32 bits.
  if (msize[0] >= (int64_t(1) << 31)) {
    if (m >= kMaxDims) return ZR_ERR_SIZE;
    int64_t w = int64_t(1) << 24;
    while (w > 1 && msize[0] % w != 0) w >>= 1;
    if (msize[0] / w >= (int64_t(1) << 31) || w == 1) return ZR_ERR_SIZE;
    for (int j = m; j > 0; --j) {
      msize[j] = msize[j - 1];
      for (int k = 0; k < kProbSlots; ++k) mst[k][j] = mst[k][j - 1];
    }
    msize[1] = msize[0] / w;
    msize[0] = w;
    for (int k = 0; k < kProbSlots; ++k) mst[k][1] = mst[k][0] * w;
    ++m;
  }
  P->n = m;
  P->active = active;
  for (int i = 0; i < m; ++i) {
    P->size[i] = msize[m - 1 - i];
    for (int k = 0; k < kProbSlots; ++k) P->st[k][i] = mst[k][m - 1 - i];
  }
  for (int i = 0; i + 1 < m; ++i)
    if (P->size[i] >= (int64_t(1) << 32)) return ZR_ERR_SIZE;
  return ZR_OK;
}

int build_ew(const Prob& P, const float* const in[3], float* const out[2], uint32_t read_mask,
             uint32_t stream_mask, int occ, EwBuild* eb) {
  EwPlan& p = eb->plan;
  p = EwPlan{};
  const int n = P.n;
  for (int k = 0; k < 3; ++k) p.in[k] = in[k];
  p.out[0] = out[0];
  p.out[1] = out[1];
  int dims[kMaxDims];
  for (int i = 0; i < n - 1; ++i) dims[i] = i;
  fill_decomp(&p.rows, P, dims, n - 1);
  for (int k = 0; k < kMaxOperands; ++k) p.inner_stride[k] = P.st[k][n - 1];
  p.stream_mask = stream_mask;

  uint64_t nrow = 1;
  for (int i = 0; i < n - 1; ++i) nrow *= uint64_t(P.size[i]);
  const uint64_t ncol = uint64_t(P.size[n - 1]);
  if (nrow >= (uint64_t(1) << 32) || ncol >= (uint64_t(1) << 31)) return ZR_ERR_SIZE;

  const void* ptrs[kMaxOperands] = {in[0], in[1], in[2], out[0] ? out[0] : out[1]};
  uint32_t slots = read_mask | (1u << kSlotOut);
  eb->vec = pick_vec(P, slots, ptrs, out[0] && out[1] ? out[1] : nullptr);
  eb->es = P.es;
  // Grids are sized with the float kernels' CTAs per SM; most 8-wide
  // bfloat16 kernels keep that figure (WideBlocks), the others one fewer.
  const uint64_t nvcol = ceil_div(ncol, eb->vec);
  const uint64_t items = nrow * nvcol;
  uint64_t ipc = items / 1216;
  ipc = std::max<uint64_t>(256, std::min<uint64_t>(2048, ipc));
  ipc = ceil_div(ipc, 256) * 256;
  uint64_t tvc = std::min<uint64_t>(nvcol, ipc);
  uint64_t trows = std::max<uint64_t>(1, ipc / tvc);
  trows = std::min<uint64_t>(trows, std::min<uint64_t>(nrow, kMaxTileRows));
  // Grid: nearby tile sizes whose CTA count fills the last wave best.
  const uint64_t wave = uint64_t(kSms) * uint64_t(occ);
  if (trows > 1 || tvc == nvcol) {
    // Rows per tile in [trows / 2, 2 trows].
    auto real = [&](uint64_t n) { return ceil_div(nrow, ceil_div(nrow, n)); };
    const uint64_t lo = ceil_div(nrow, std::min<uint64_t>({2 * trows, nrow, kMaxTileRows}));
    const uint64_t hi = ceil_div(nrow, std::max<uint64_t>(1, trows / 2));
    const uint64_t n = fit_waves(ceil_div(nrow, trows), lo, hi, ceil_div(nvcol, tvc), wave, real);
    trows = ceil_div(nrow, n);
  } else {
    // One row per tile: vectors per tile in [tvc / 2, 2 tvc], multiples of
    // 128 (2 KB of each operand).
    auto width = [&](uint64_t n) {
      return std::min<uint64_t>(nvcol, ceil_div(ceil_div(nvcol, n), 128) * 128);
    };
    auto real = [&](uint64_t n) { return ceil_div(nvcol, width(n)); };
    const uint64_t lo = ceil_div(nvcol, std::min<uint64_t>(nvcol, 2 * tvc));
    const uint64_t hi = ceil_div(nvcol, std::max<uint64_t>(128, tvc / 2));
    const uint64_t n = fit_waves(ceil_div(nvcol, tvc), lo, hi, nrow, wave, real);
    tvc = width(n);
  }
  p.nrow = uint32_t(nrow);
  p.ncol = uint32_t(ncol);
  p.nvcol = uint32_t(nvcol);
  p.tile_vcols = uint32_t(tvc);
  p.tile_rows = uint32_t(trows);
  p.col_tiles = uint32_t(ceil_div(nvcol, tvc));
  p.col_tiles_div = make_fastdiv(p.col_tiles);
  p.tile_vcols_div = make_fastdiv(p.tile_vcols);
  p.items_per_cta = uint32_t(trows * tvc);
  const uint64_t ncta = ceil_div(nrow, trows) * p.col_tiles;
  if (ncta >= (uint64_t(1) << 31)) return ZR_ERR_SIZE;
  p.n_cta = uint32_t(ncta);
  // Flat plan for at most one outer dim: no offset table; CTAs of whole
  // 1024-item batches (the kernel's 4 loads in flight x 256 threads), fewer
  // per CTA (down to one item per thread) when that is what fills the GPU.
  if (n <= 2 && items <= kFlatMaxItems) {
    uint64_t ipc = kFlatBatch;
    while (ipc > kThreads && ceil_div(items, ipc) < wave) ipc /= 2;
    p.flat = 1;
    p.nitems = uint32_t(items);
    p.nvcol_div = make_fastdiv(p.nvcol);
    p.items_per_cta = uint32_t(ipc);
    p.tile_rows = 0;
    p.tile_vcols = 0;
    p.col_tiles = 0;
    p.n_cta = uint32_t(ceil_div(items, ipc));
  }
  return ZR_OK;
}

int build_red(const Prob& P, int xslot, const float* g, const float* a, const float* b,
              uint32_t read_mask, uint32_t stream_mask, float* x_out, float* d_out,
              int vec_override, int occ, int occ_cl_kept, int occ_cl_red, RedBuild* rb,
              bool post) {
  RedPlan& p = rb->plan;
  p = RedPlan{};
  const int n = P.n;
  p.g = g;
  p.a = a;
  p.b = b;
  p.x_final = x_out;
  p.d_out = d_out;
  p.stream_mask = stream_mask;
  p.scale = 1.0f;
  int kd[kMaxDims], rd[kMaxDims];
  int nk = 0, nr = 0;
  uint64_t n_kept = 1, n_red = 1;
  for (int d = 0; d < n - 1; ++d) {
    if (P.st[xslot][d] != 0) { kd[nk++] = d; n_kept *= uint64_t(P.size[d]); }
    else { rd[nr++] = d; n_red *= uint64_t(P.size[d]); }
  }
  fill_decomp(&p.kept, P, kd, nk);
  fill_decomp(&p.red, P, rd, nr);
  for (int k = 0; k < kMaxOperands; ++k) p.inner_stride[k] = P.st[k][n - 1];
  const uint64_t ncol = uint64_t(P.size[n - 1]);
  p.inner_kept = P.st[xslot][n - 1] != 0 ? 1 : 0;
  if (n_kept >= (uint64_t(1) << 32) || n_red >= (uint64_t(1) << 32) ||
      ncol >= (uint64_t(1) << 31))
    return ZR_ERR_SIZE;
  p.n_kept = uint32_t(n_kept);
  p.n_red = uint32_t(n_red);
  p.ncol = uint32_t(ncol);
  p.nout = p.inner_kept ? n_kept * ncol : n_kept;

  const void* ptrs[kMaxOperands] = {g, a, b, d_out};
  uint32_t slots = (read_mask & 7u) | (d_out ? (1u << kSlotOut) : 0u);
  rb->es = P.es;
  // The reduced gradient's kept outer strides are multiples of ncol, so its
  // rows stay aligned; the workspace is 16-byte aligned by contract.
  rb->vec = vec_override ? vec_override
                         : pick_vec(P, slots, ptrs, p.inner_kept ? static_cast<const void*>(x_out)
                                                                 : nullptr);
  // 8-wide bfloat16 mul/div reductions with the inner dim kept run one CTA
  // per SM fewer than the float kernel (red_wide_occ).
  if (rb->vec == 8 && p.inner_kept && occ < 4) occ = wide_occ(occ);
  const uint32_t vec = uint32_t(rb->vec);
  const uint64_t nvcol = ceil_div(ncol, vec);
  p.nvcol = uint32_t(nvcol);

  const uint64_t total = n_kept * n_red * ncol;
  const uint64_t E = elems_per_cta_target(total);
  // Partial slots are capped so that their write + read stays within about
  // 3% of the input stream, and at 4096 for the second pass.
  uint64_t cap = total / (64 * std::max<uint64_t>(1, p.nout));
  cap = std::max<uint64_t>(1, std::min<uint64_t>(4096, cap));

  const uint32_t tx_wide = pick_tx(nvcol);
  uint32_t tx = tx_wide;
  uint64_t rows, vcols;
  const uint64_t wave = uint64_t(kSms) * uint64_t(occ);
  if (p.inner_kept) {
    // Narrow the column lanes while that adds CTAs the slot cap would
    // otherwise forbid.
    while (tx > 32) {
      const uint64_t ty = kThreads / tx;
      const uint64_t ctas = n_kept * ceil_div(nvcol, tx) * std::min<uint64_t>(cap, ceil_div(n_red, ty));
      if (ctas >= 1216) break;
      tx /= 2;
    }
    auto rows_for = [&](uint32_t t) {
      uint64_t r = ceil_div(E, uint64_t(t) * vec);
      r = std::max<uint64_t>(r, ceil_div(n_red, cap));
      return std::min<uint64_t>(r, n_red);
    };
    rows = rows_for(tx);
    // Grid: over column-lane widths from 32 to the widest, and row blocks
    // in [n0 / 2, 2 n0], the shape whose CTA count fills the last wave best;
    // one partial slot (no combine pass) is worth 0.02 of fill, and a plan
    // with one slot keeps it.
    auto real = [&](uint64_t n) { return ceil_div(n_red, ceil_div(n_red, n)); };
    auto score = [&](uint32_t t, uint64_t n) {
      const uint64_t nb = real(n);
      return wave_fill(n_kept * ceil_div(nvcol, t) * nb, wave) - (nb > 1 ? 0.02 : 0.0);
    };
    uint32_t best_tx = tx;
    uint64_t best_n = ceil_div(n_red, rows);
    double best = score(tx, best_n);
    for (uint32_t t = tx_wide; t >= 1; t /= 2) {
      if (t < 32 && t != tx_wide) break;
      const uint64_t n0 = ceil_div(n_red, rows_for(t));
      const uint64_t lo = std::max<uint64_t>(1, n0 / 2);
      const uint64_t hi = n0 == 1 ? 1 : std::min<uint64_t>({2 * n0, cap, n_red});
      const uint64_t F = n_kept * ceil_div(nvcol, t);
      const uint64_t n = fit_waves(n0, lo, std::max(hi, lo), F, wave, real);
      const double sc = score(t, n);
      if (sc > best + 1e-9) { best = sc; best_tx = t; best_n = n; }
    }
    tx = best_tx;
    rows = ceil_div(n_red, best_n);
    // 8-wide vectors with every reduced row in one block: 64 column lanes
    // (4 row lanes), so that each thread streams a quarter of the rows, as
    // the 4-wide plans do, and a staged CTA's pipeline runs for more passes
    // than it takes to fill (c4 in bf16, backward add: 69.2 -> 66.3 us, with
    // half the CTAs).
    if (vec == 8 && best_n == 1 && tx < 64 && tx_wide >= 64) tx = 64;
    vcols = tx;
  } else {
    if (nvcol * vec >= E) {
      vcols = ceil_div(ceil_div(E, vec), tx) * tx;
      rows = 1;
    } else {
      vcols = ceil_div(nvcol, tx) * tx;
      rows = std::max<uint64_t>(1, E / (nvcol * vec));
      rows = std::min<uint64_t>(rows, n_red);
    }
    for (;;) {
      const uint64_t slots_now = ceil_div(n_red, rows) * ceil_div(nvcol, vcols);
      if (slots_now <= cap) break;
      if (rows < n_red) rows = std::min<uint64_t>(n_red, rows * 2);
      else vcols *= 2;
    }
    // Grid: row blocks (or, with one row per block, column blocks in
    // multiples of tx vectors) whose CTA count fills the last wave best,
    // keeping the slots within the cap; a plan with one slot keeps it.
    const uint64_t n_cb = ceil_div(nvcol, vcols);
    if (ceil_div(n_red, rows) * n_cb == 1) {
      // one slot: no combine pass
    } else if (rows > 1 || n_cb == 1) {
      auto real = [&](uint64_t n) { return ceil_div(n_red, ceil_div(n_red, n)); };
      const uint64_t n0 = ceil_div(n_red, rows);
      const uint64_t lo = std::max<uint64_t>(1, n0 / 2);
      const uint64_t hi = std::max(lo, std::min<uint64_t>({2 * n0, n_red, cap / n_cb}));
      const uint64_t n = fit_waves(n0, lo, hi, n_kept * n_cb, wave, real);
      rows = ceil_div(n_red, n);
    } else {
      auto width = [&](uint64_t n) {
        return std::min<uint64_t>(ceil_div(nvcol, tx) * tx, ceil_div(ceil_div(nvcol, n), tx) * tx);
      };
      auto real = [&](uint64_t n) { return ceil_div(nvcol, width(n)); };
      const uint64_t lo = std::max<uint64_t>(1, n_cb / 2);
      const uint64_t hi = std::max(lo, std::min<uint64_t>(2 * n_cb, cap / std::max<uint64_t>(1, n_red)));
      const uint64_t n = fit_waves(n_cb, lo, hi, n_kept * n_red, wave, real);
      vcols = width(n);
    }
  }
  // Combine-free alternative: when the plan above needs partial slots and
  // 16-byte vectors apply, let the CTAs of one output tile form a cluster
  // (at most kMaxCluster CTAs) that covers every reduced row, so the tile's
  // total is formed on chip and no second pass runs.  Taken, widest column
  // lanes first, when its grid is resident at once (cluster_wave) and fills
  // three quarters of a wave or has at least as many CTAs as the plan above.
  p.cluster = 1;
  const uint64_t std_slots = p.inner_kept ? ceil_div(n_red, rows)
                                          : ceil_div(n_red, rows) * ceil_div(nvcol, vcols);
  const uint64_t std_ctas = n_kept * ceil_div(n_red, rows) * ceil_div(nvcol, vcols);
  const int occ_cl = p.inner_kept ? occ_cl_kept : occ_cl_red;
  if (occ_cl > 0 && vec == 4 && P.es == 4 && std_slots > 1) {
    const uint64_t wave_cl = uint64_t(kSms) * uint64_t(occ_cl);
    // Inner dim kept: column lanes from the widest down to 8 (128-byte row
    // segments), tiles = kept index x column block; reduced: tiles = kept
    // indices, each CTA covering whole rows.
    for (uint32_t t = p.inner_kept ? tx_wide : pick_tx(nvcol); t >= 8; t /= 2) {
      const uint64_t vc = p.inner_kept ? t : ceil_div(nvcol, t) * t;
      const uint64_t tiles = n_kept * ceil_div(nvcol, vc);
      uint64_t c_max = std::min<uint64_t>({kMaxCluster, wave_cl / tiles, n_red});
      while (c_max > 1 && tiles * c_max > cluster_wave(wave_cl, c_max)) --c_max;
      if (c_max >= 1) {
        const uint64_t r = ceil_div(n_red, c_max);
        const uint64_t c = ceil_div(n_red, r);
        const uint64_t need = std::min<uint64_t>(ceil_div(3 * wave_cl, 4), std_ctas);
        if (c >= 2 && tiles * c >= need && r >= kThreads / t) {
          tx = t;
          vcols = vc;
          rows = r;
          p.cluster = uint32_t(c);
          break;
        }
      }
      if (!p.inner_kept) break;
    }
  }
  p.tx = tx;
  p.ty = kThreads / tx;
  p.rows_per_blk = uint32_t(rows);
  p.vcols_per_blk = uint32_t(vcols);
  p.n_rblk = uint32_t(ceil_div(n_red, rows));
  p.n_cblk = uint32_t(ceil_div(nvcol, vcols));
  p.n_cblk_div = make_fastdiv(p.n_cblk);
  p.n_rblk_div = make_fastdiv(p.n_rblk);
  p.nslots = p.cluster > 1 ? 1 : (p.inner_kept ? p.n_rblk : p.n_rblk * p.n_cblk);
  p.cluster_div = make_fastdiv(p.cluster);
  const uint64_t ncta = n_kept * p.n_rblk * uint64_t(p.n_cblk);
  if (ncta >= (uint64_t(1) << 31)) return ZR_ERR_SIZE;
  p.n_cta = uint32_t(ncta);
  const uint64_t ws_floats = uint64_t(p.nslots) * p.nout + (post ? p.nout : 0);
  rb->ws_bytes = p.nslots > 1 ? ((ws_floats * sizeof(float) + 255) / 256) * 256 : 0;

  // cp.async staging when every streamed input (g, and a or b unless it is
  // the reduced gradient's own input, read once per thread) is read in
  // 16-byte vectors with unit inner stride, and the grid runs at least two
  // waves: three batches in flight where the CTAs per SM of the kernel still
  // fit in shared memory, else two.  (Measured on GB300: c4's backward
  // 186 -> 178 us and 121 -> 118 us, c4 in bf16 111 -> 102 us and
  // 77 -> 71 us; single-wave grids, whose CTAs each stream one long range,
  // measured slower staged: c5a's backward 22.9 -> 24.3 us.)
  p.stages = 0;
  p.stage_ns = 0;
  const uint64_t cta_wave = uint64_t(kSms) * uint64_t(p.cluster > 1 ? occ_cl : occ);
  if (uint32_t(rb->vec) * uint32_t(P.es) == 16 && uint64_t(p.n_cta) >= 2 * cta_wave) {
    const uint32_t own = xslot == kSlotXA ? 2u : (xslot == kSlotXB ? 4u : 0u);  // a's or b's slot
    const uint32_t streamed = ((read_mask & 7u) & ~own) | 1u;
    bool unit = true;
    uint32_t ns = 0;
    for (int k = 0; k < 3; ++k)
      if (streamed & (1u << k)) {
        ++ns;
        if (P.st[k][n - 1] != 1) unit = false;
      }
    const uint32_t cta_occ = p.cluster > 1 ? uint32_t(occ_cl) : uint32_t(occ);
    if (unit && ns <= 2) {
      for (uint32_t st = 3; st >= 2; --st) {
        const uint64_t bytes = red_smem_bytes(p, rb->vec, st, ns);
        if (cta_occ * (bytes + kSmemReservedPerCta) <= kSmemPerSm) {
          p.stages = st;
          p.stage_ns = ns;
          break;
        }
      }
    }
  }

  CombinePlan& c = rb->comb;
  c = CombinePlan{};
  c.nout = p.nout;
  c.split = p.nout;
  c.nslots = p.nslots;
  c.out = x_out;
  c.scale = 1.0f;
  c.post = post && p.nslots > 1 ? 1u : 0u;
  combine_layout(&c);
  return ZR_OK;
}

int build_chain(const Prob& P, const float* g, const float* a, const float* b, const float* c,
                bool c_scalar, float* grad_a, float* grad_b, float* grad_c, uint32_t stream_mask,
                int vec_override, ChainBuild* cb, bool div1, bool div2) {
  *cb = ChainBuild{};
  // c is read with b's offsets (same shape, both dense), so it needs b's
  // 16-byte alignment; a single-element c is read as a scalar.
  if (!c_scalar && vec_override == 0 && reinterpret_cast<uintptr_t>(c) % 16 != 0) return 1;
  RedBuild rb;
  const int rc = build_red(P, kSlotXB, g, a, b, 7u, stream_mask & 7u, grad_b, grad_a,
                           vec_override, kOccChain, 0, 0, &rb, div1);
  if (rc) return rc;
  if (rb.vec != 4 || !rb.plan.inner_kept) return 1;
  ChainPlan& cp = cb->plan;
  cp.r = rb.plan;
  cp.c = c;
  cp.c_final = grad_c;
  cp.c_scalar = c_scalar ? 1 : 0;
  cb->comb_b = rb.comb;
  cb->ws_b_bytes = rb.ws_bytes;
  CombinePlan& cc = cb->comb_c;
  cc = CombinePlan{};
  if (c_scalar) {
    cc.nout = 1;
    cc.split = 1;
    cc.nslots = rb.plan.n_cta;
    cc.out = grad_c;
    cc.scale = 1.0f;
    // Division by c: the per-CTA partials are followed by the factor -1/c^2.
    cc.post = div2 && rb.plan.n_cta > 1 ? 1u : 0u;
    combine_layout(&cc);
    cb->ws_c_bytes = rb.plan.n_cta > 1
                         ? ((uint64_t(rb.plan.n_cta + (div2 ? 1 : 0)) * 4 + 255) / 256) * 256
                         : 0;
  } else if (rb.plan.nslots > 1) {
    // One second pass over [nslots][2 nout]: grad_b, then grad_c; with a
    // division in the chain, a row of per-output factors follows the slots.
    CombinePlan& c2 = cb->comb_b;
    c2.nout = 2 * rb.plan.nout;
    c2.split = rb.plan.nout;
    c2.out2 = grad_c;
    c2.post = (div1 || div2) ? 1u : 0u;
    combine_layout(&c2);
    cb->ws_b_bytes =
        ((uint64_t(rb.plan.nslots + c2.post) * c2.nout * 4 + 255) / 256) * 256;
  }
  return ZR_OK;
}

std::string describe_chain(const ChainBuild& cb) {
  RedBuild rb;
  rb.plan = cb.plan.r;
  rb.comb = cb.comb_b;
  rb.vec = 4;
  rb.ws_bytes = cb.ws_b_bytes;
  std::string r = describe_red(rb);
  char buf[160];
  std::snprintf(buf, sizeof(buf), ",\"c_scalar\":%u,\"c_slots\":%u,\"ws_c_bytes\":%zu}",
                cb.plan.c_scalar, cb.comb_c.nslots, cb.ws_c_bytes);
  r.pop_back();
  r.replace(r.find("\"kernel\":\"reduce\""), 17, "\"kernel\":\"chain\"");
  return r + buf;
}

int build_tr(const Prob& P, const float* a, const float* b, float* out, TrPlan* tp) {
  const int n = P.n;
  const int q = n - 1;
  if (n < 2 || P.st[kSlotOut][q] != 1) return 1;
  int xs = -1, pd = -1;
  for (int k = 0; k < 2 && xs < 0; ++k) {
    if (P.st[k][q] == 0 || P.st[k][q] == 1) continue;
    for (int d = 0; d < q; ++d)
      if (P.st[k][d] == 1) { xs = k; pd = d; break; }
  }
  if (xs < 0) return 1;
  const int ys = 1 - xs;
  if (P.size[pd] >= (int64_t(1) << 31) || P.size[q] >= (int64_t(1) << 31)) return 1;
  TrPlan& p = *tp;
  p = TrPlan{};
  p.x = xs == 0 ? a : b;
  p.y = xs == 0 ? b : a;
  p.out = out;
  p.x_is_a = xs == 0 ? 1 : 0;
  // Batch dims in row-major order, remapped to slots x=0, y=1, out=3.
  int dims[kMaxDims];
  int nd = 0;
  uint64_t nbatch = 1;
  for (int d = 0; d < q; ++d)
    if (d != pd) { dims[nd++] = d; nbatch *= uint64_t(P.size[d]); }
  p.batch.n = nd;
  for (int i = 0; i < kMaxDims; ++i) {
    p.batch.div[i] = make_fastdiv(1);
    for (int k = 0; k < kMaxOperands; ++k) p.batch.stride[k][i] = 0;
  }
  for (int i = 0; i < nd; ++i) {
    const int d = dims[nd - 1 - i];
    p.batch.div[i] = make_fastdiv(uint32_t(P.size[d]));
    p.batch.stride[0][i] = P.st[xs][d];
    p.batch.stride[1][i] = P.st[ys][d];
    p.batch.stride[kSlotOut][i] = P.st[kSlotOut][d];
  }
  p.xs_q = P.st[xs][q];
  p.ys_p = P.st[ys][pd];
  p.ys_q = P.st[ys][q];
  p.os_p = P.st[kSlotOut][pd];
  p.np = uint32_t(P.size[pd]);
  p.nq = uint32_t(P.size[q]);
  p.n_pt = uint32_t(ceil_div(p.np, kTrP));
  p.n_qt = uint32_t(ceil_div(p.nq, kTrTile));
  p.n_qt_div = make_fastdiv(p.n_qt);
  p.n_pt_div = make_fastdiv(p.n_pt);
  const uint64_t ncta = nbatch * p.n_pt * p.n_qt;
  if (nbatch >= (uint64_t(1) << 32) || ncta >= (uint64_t(1) << 31)) return 1;
  p.n_cta = uint32_t(ncta);
  // 16-byte loads of x along p and stores of out along q.
  bool v = reinterpret_cast<uintptr_t>(p.x) % 16 == 0 && p.xs_q % 4 == 0 &&
           reinterpret_cast<uintptr_t>(p.out) % 16 == 0 && p.os_p % 4 == 0;
  for (int i = 0; i < nd; ++i)
    v = v && p.batch.stride[0][i] % 4 == 0 && p.batch.stride[kSlotOut][i] % 4 == 0;
  p.vec_ok = v ? 1 : 0;
  return ZR_OK;
}

std::string describe_tr(const TrPlan& p) {
  char buf[512];
  std::snprintf(buf, sizeof(buf),
                "{\"kernel\":\"transpose\",\"x_is_a\":%u,\"np\":%u,\"nq\":%u,\"batch_dims\":%d,"
                "\"xs_q\":%lld,\"ctas\":%u}",
                p.x_is_a, p.np, p.nq, p.batch.n, (long long)p.xs_q, p.n_cta);
  return buf;
}

std::string describe_ew(const EwBuild& eb) {
  const EwPlan& p = eb.plan;
  char buf[1024];
  std::snprintf(buf, sizeof(buf),
                "{\"kernel\":\"%s\",\"vec\":%d,\"nrow\":%u,\"ncol\":%u,\"row_dims\":%d,"
                "\"inner_stride\":[%lld,%lld,%lld,%lld],\"tile_rows\":%u,\"tile_vcols\":%u,"
                "\"items_per_cta\":%u,\"ctas\":%u,\"stream_mask\":%u}",
                eb.gelu_tab ? "gelu_table" : p.flat ? "flat" : "elementwise", eb.vec, p.nrow, p.ncol, p.rows.n,
                (long long)p.inner_stride[0], (long long)p.inner_stride[1],
                (long long)p.inner_stride[2], (long long)p.inner_stride[3], p.tile_rows,
                p.tile_vcols, p.items_per_cta, p.n_cta, p.stream_mask);
  return buf;
}

std::string describe_red(const RedBuild& rb) {
  const RedPlan& p = rb.plan;
  char buf[1024];
  std::snprintf(buf, sizeof(buf),
                "{\"kernel\":\"reduce\",\"vec\":%d,\"inner_kept\":%u,\"n_kept\":%u,\"n_red\":%u,"
                "\"ncol\":%u,\"kept_dims\":%d,\"red_dims\":%d,\"tx\":%u,\"ty\":%u,"
                "\"rows_per_blk\":%u,\"vcols_per_blk\":%u,\"n_rblk\":%u,\"n_cblk\":%u,"
                "\"nslots\":%u,\"nout\":%llu,\"ctas\":%u,\"ws_bytes\":%zu,\"dense_out\":%d,"
                "\"cluster\":%u,\"stages\":%u,\"stage_ns\":%u}",
                rb.vec, p.inner_kept, p.n_kept, p.n_red, p.ncol, p.kept.n, p.red.n, p.tx, p.ty,
                p.rows_per_blk, p.vcols_per_blk, p.n_rblk, p.n_cblk, p.nslots,
                (unsigned long long)p.nout, p.n_cta, rb.ws_bytes, p.d_out ? 1 : 0, p.cluster,
                p.stages, p.stage_ns);
  return buf;
}

}  // namespace zr

namespace zr {

namespace {

// Fill a decomposition from an explicit dim list (outer to inner), each with
// a size and up to three operand strides.
struct DimSpec {
  uint64_t size;
  int64_t st[3];  // operand slots 0..2
};
void fill_from_specs(Decomp* dc, const DimSpec* dims, int nd) {
  dc->n = nd;
  for (int i = 0; i < kMaxDims; ++i) {
    dc->div[i] = make_fastdiv(1);
    for (int k = 0; k < kMaxOperands; ++k) dc->stride[k][i] = 0;
  }
  for (int i = 0; i < nd; ++i) {
    const DimSpec& d = dims[nd - 1 - i];
    dc->div[i] = make_fastdiv(static_cast<uint32_t>(d.size));
    for (int k = 0; k < 3; ++k) dc->stride[k][i] = d.st[k];
  }
}

}  // namespace

int build_sab(const Prob& P, const float* g, const float* a, const float* b, float* grad_a,
              float* grad_b, uint32_t read_mask, SabBuild* sb, bool post) {
  const int n = P.n;
  if (n < 2 || !grad_a || !grad_b) return 1;
  const int I = n - 1;
  // Inner dim kept by both, unit stride for every operand read.
  if (P.st[kSlotXA][I] == 0 || P.st[kSlotXB][I] == 0) return 1;
  for (int k = 0; k < 3; ++k)
    if ((read_mask & (1u << k)) && P.st[k][I] != 1) return 1;
  const uint64_t ncol = uint64_t(P.size[I]);
  if (ncol % 4 != 0) return 1;
  const uint64_t nvc = ncol / 4;
  if (nvc > 32 || (nvc & (nvc - 1)) != 0) return 1;
  const void* ptrs[3] = {g, a, b};
  for (int k = 0; k < 3; ++k) {
    if (!(read_mask & (1u << k))) continue;
    if (reinterpret_cast<uintptr_t>(ptrs[k]) % 16 != 0) return 1;
    for (int d = 0; d < I; ++d)
      if (P.st[k][d] % 4 != 0) return 1;
  }
  // Every outer dim is kept by exactly one input.
  int adims[kMaxDims], bdims[kMaxDims];
  int na = 0, nb = 0;
  uint64_t n_alpha = 1, n_beta = 1;
  for (int d = 0; d < I; ++d) {
    const bool ka = P.st[kSlotXA][d] != 0, kb = P.st[kSlotXB][d] != 0;
    if (ka == kb) return 1;
    if (ka) { adims[na++] = d; n_alpha *= uint64_t(P.size[d]); }
    else { bdims[nb++] = d; n_beta *= uint64_t(P.size[d]); }
  }
  if (na == 0 || nb == 0 || n_beta > 4096) return 1;
  // Rows per tile: from the innermost A dims outwards, at most 2048/nvc rows,
  // splitting one dim by its largest fitting divisor.
  const uint64_t ta_max = 2048 / nvc;
  DimSpec inner[kMaxDims + 1], outer[kMaxDims + 1];
  int n_in = 0, n_out = 0;
  uint64_t ta = 1;
  int i = na - 1;
  for (; i >= 0; --i) {
    const int d = adims[i];
    const uint64_t s = uint64_t(P.size[d]);
    if (ta * s <= ta_max) {
      inner[n_in++] = {s, {P.st[0][d], P.st[1][d], P.st[2][d]}};
      ta *= s;
      continue;
    }
    uint64_t f = ta_max / ta;
    while (f > 1 && s % f != 0) --f;
    if (f > 1) {
      inner[n_in++] = {f, {P.st[0][d], P.st[1][d], P.st[2][d]}};
      outer[n_out++] = {s / f, {P.st[0][d] * int64_t(f), P.st[1][d] * int64_t(f),
                                P.st[2][d] * int64_t(f)}};
      ta *= f;
    } else {
      outer[n_out++] = {s, {P.st[0][d], P.st[1][d], P.st[2][d]}};
    }
    --i;
    break;
  }
  for (; i >= 0; --i) {
    const int d = adims[i];
    outer[n_out++] = {uint64_t(P.size[d]), {P.st[0][d], P.st[1][d], P.st[2][d]}};
  }
  const uint64_t rows_x_vec = ta * nvc;
  if (rows_x_vec < uint64_t(kSabThreads) || rows_x_vec > 2048 ||
      (rows_x_vec & (rows_x_vec - 1)) != 0)
    return 1;
  if (n_in > kMaxDims || n_out > kMaxDims) return 1;
  // inner[] / outer[] were collected inner-to-outer; reverse into row-major.
  std::reverse(inner, inner + n_in);
  std::reverse(outer, outer + n_out);
  DimSpec beta[kMaxDims];
  for (int j = 0; j < nb; ++j) {
    const int d = bdims[j];
    beta[j] = {uint64_t(P.size[d]), {P.st[0][d], P.st[1][d], P.st[2][d]}};
  }
  const uint64_t n_tiles = n_alpha / ta;
  // Steps are indexed in 32 bits; the slot count is found by a walk over tiles.
  if (n_tiles > (uint64_t(1) << 22) || n_tiles * n_beta >= (uint64_t(1) << 32)) return 1;

  SabPlan& p = sb->plan;
  p = SabPlan{};
  p.g = g;
  p.a = (read_mask & 2) ? a : nullptr;
  p.b = (read_mask & 4) ? b : nullptr;
  fill_from_specs(&p.a_outer, outer, n_out);
  fill_from_specs(&p.a_inner, inner, n_in);
  fill_from_specs(&p.beta, beta, nb);
  p.ncol = uint32_t(ncol);
  p.nvc = uint32_t(nvc);
  p.ta = uint32_t(ta);
  p.n_tiles = uint32_t(n_tiles);
  p.n_beta = uint32_t(n_beta);
  p.n_beta_div = make_fastdiv(p.n_beta);
  p.total_steps = n_tiles * n_beta;
  p.grid = uint32_t(std::min<uint64_t>(kSabGrid, p.total_steps));
  p.n_a = n_alpha * ncol;
  p.n_b = n_beta * ncol;
  uint32_t smax = 1;
  for (uint64_t t = 0; t < n_tiles; ++t) {
    const uint32_t c0 = sab_owner(p, t * n_beta);
    const uint32_t c1 = sab_owner(p, t * n_beta + n_beta - 1);
    smax = std::max(smax, c1 - c0 + 1);
  }
  p.slots_a = smax;
  // grad_b's per-warp partials wait in a ring of (ring + 1) steps, each
  // [warps][ncol] plus the step's b factors [ncol]; the largest ring that
  // fits (at most one column-step per thread per pass) is taken.
  const uint64_t fixed = uint64_t(kSabStages) * (ta + 1) * ncol * 4 + 2 * ta * 8 + 2 * n_beta * 8;
  uint64_t ring = kSabThreads / ncol, smem = 0;
  for (; ring >= 1; ring /= 2) {
    smem = fixed + (ring + 1) * (kSabThreads / 32 + 1) * ncol * 4;
    if (smem <= 220 * 1024) break;
  }
  if (ring < 1) return 1;
  p.ring = uint32_t(ring);
  p.smem_bytes = uint32_t(smem);
  sb->rpt = int(rows_x_vec / kSabThreads);
  sb->ws_a_bytes = ((uint64_t(p.slots_a) * p.n_a * 4 + 255) / 256) * 256;
  // grad_b's region: its partial slots, then (post) one factor per output.
  sb->ws_b_bytes = ((uint64_t(p.n_tiles + (post ? 1 : 0)) * p.n_b * 4 + 255) / 256) * 256;
  CombinePlan* cs[2] = {&sb->comb_a, &sb->comb_b};
  const uint64_t nouts[2] = {p.n_a, p.n_b};
  const uint32_t nsl[2] = {p.slots_a, p.n_tiles};
  float* outs[2] = {grad_a, grad_b};
  for (int w = 0; w < 2; ++w) {
    CombinePlan& c = *cs[w];
    c = CombinePlan{};
    c.nout = nouts[w];
    c.split = nouts[w];
    c.nslots = nsl[w];
    c.out = outs[w];
    c.scale = 1.0f;
    c.post = (w == 1 && post) ? 1u : 0u;
    combine_layout(&c);
  }
  return ZR_OK;
}

int build_sabf(const Prob& P, const float* a, const float* b, float* out, SabFPlan* sp, int* rpt) {
  const int n = P.n;
  if (n < 2) return 1;
  const int I = n - 1;
  // Slots in P: a = 0, b = 1, out = 3.
  if (P.st[0][I] != 1 || P.st[1][I] != 1 || P.st[kSlotOut][I] != 1) return 1;
  const uint64_t ncol = uint64_t(P.size[I]);
  if (ncol % 4 != 0) return 1;
  const uint64_t nvc = ncol / 4;
  if (nvc > 32 || (nvc & (nvc - 1)) != 0) return 1;
  const void* ptrs[3] = {a, b, out};
  const int slots[3] = {0, 1, kSlotOut};
  for (int k = 0; k < 3; ++k) {
    if (reinterpret_cast<uintptr_t>(ptrs[k]) % 16 != 0) return 1;
    for (int d = 0; d < I; ++d)
      if (P.st[slots[k]][d] % 4 != 0) return 1;
  }
  int adims[kMaxDims], bdims[kMaxDims];
  int na = 0, nb = 0;
  uint64_t n_alpha = 1, n_beta = 1;
  for (int d = 0; d < I; ++d) {
    const bool va = P.st[0][d] != 0, vb = P.st[1][d] != 0;
    if (va == vb) return 1;
    if (va) { adims[na++] = d; n_alpha *= uint64_t(P.size[d]); }
    else { bdims[nb++] = d; n_beta *= uint64_t(P.size[d]); }
  }
  if (na == 0 || nb == 0) return 1;
  // Rows per tile from the innermost A dims (one of them possibly split),
  // at most 2048/nvc rows: 256 threads x up to 8 float4 rows each.
  const uint64_t ta_max = 2048 / nvc;
  DimSpec inner[kMaxDims + 1], outer[kMaxDims + 1];
  int n_in = 0, n_out = 0;
  uint64_t ta = 1;
  auto spec = [&](int d, uint64_t size, int64_t mult) {
    return DimSpec{size, {P.st[kSlotOut][d] * mult, P.st[0][d] * mult, P.st[1][d] * mult}};
  };
  int i = na - 1;
  for (; i >= 0; --i) {
    const int d = adims[i];
    const uint64_t s = uint64_t(P.size[d]);
    if (ta * s <= ta_max) { inner[n_in++] = spec(d, s, 1); ta *= s; continue; }
    uint64_t f = ta_max / ta;
    while (f > 1 && s % f != 0) --f;
    if (f > 1) {
      inner[n_in++] = spec(d, f, 1);
      outer[n_out++] = spec(d, s / f, int64_t(f));
      ta *= f;
    } else {
      outer[n_out++] = spec(d, s, 1);
    }
    --i;
    break;
  }
  for (; i >= 0; --i) outer[n_out++] = spec(adims[i], uint64_t(P.size[adims[i]]), 1);
  const uint64_t rows_x_vec = ta * nvc;
  if (rows_x_vec < 256 || rows_x_vec > 2048 || (rows_x_vec & (rows_x_vec - 1)) != 0) return 1;
  if (n_in > kMaxDims || n_out > kMaxDims) return 1;
  std::reverse(inner, inner + n_in);
  std::reverse(outer, outer + n_out);
  DimSpec beta[kMaxDims];
  for (int j = 0; j < nb; ++j) {
    const int d = bdims[j];
    beta[j] = {uint64_t(P.size[d]), {P.st[kSlotOut][d], 0, P.st[1][d]}};
  }
  const uint64_t n_tiles = n_alpha / ta;
  if (n_tiles >= (uint64_t(1) << 31) || n_beta >= (uint64_t(1) << 31)) return 1;
  SabFPlan& p = *sp;
  p = SabFPlan{};
  p.a = a;
  p.b = b;
  p.out = out;
  fill_from_specs(&p.a_outer, outer, n_out);
  fill_from_specs(&p.a_inner, inner, n_in);
  fill_from_specs(&p.beta, beta, nb);
  p.ncol = uint32_t(ncol);
  p.nvc = uint32_t(nvc);
  p.ta = uint32_t(ta);
  p.n_tiles = uint32_t(n_tiles);
  p.n_beta = uint32_t(n_beta);
  // About 512 KB written per CTA, and at least ~8 CTAs per SM in total.
  uint64_t chunk = std::max<uint64_t>(1, (512 * 1024) / (ta * ncol * 4));
  while (chunk > 1 && n_tiles * ceil_div(n_beta, chunk) < 1216) chunk /= 2;
  chunk = std::min<uint64_t>(chunk, n_beta);
  {
    // Grid: chunks in [chunk / 2, 2 chunk] whose CTA count fills the last
    // wave best.
    auto real = [&](uint64_t n) { return ceil_div(n_beta, ceil_div(n_beta, n)); };
    const uint64_t n0 = ceil_div(n_beta, chunk);
    const uint64_t lo = ceil_div(n_beta, std::min<uint64_t>(n_beta, 2 * chunk));
    const uint64_t hi = ceil_div(n_beta, std::max<uint64_t>(1, chunk / 2));
    const uint64_t n = fit_waves(n0, lo, hi, n_tiles, uint64_t(kSms) * kOccSabf, real);
    chunk = ceil_div(n_beta, n);
  }
  p.beta_chunk = uint32_t(chunk);
  p.n_bc = uint32_t(ceil_div(n_beta, p.beta_chunk));
  p.n_bc_div = make_fastdiv(p.n_bc);
  const uint64_t ncta = n_tiles * p.n_bc;
  if (ncta >= (uint64_t(1) << 31)) return 1;
  p.n_cta = uint32_t(ncta);
  *rpt = int(rows_x_vec / 256);
  return ZR_OK;
}

std::string describe_sabf(const SabFPlan& p, int rpt) {
  char buf[512];
  std::snprintf(buf, sizeof(buf),
                "{\"kernel\":\"sab_fwd\",\"ncol\":%u,\"ta\":%u,\"rpt\":%d,\"n_tiles\":%u,"
                "\"n_beta\":%u,\"beta_chunk\":%u,\"ctas\":%u}",
                p.ncol, p.ta, rpt, p.n_tiles, p.n_beta, p.beta_chunk, p.n_cta);
  return buf;
}

std::string describe_sab(const SabBuild& sb) {
  const SabPlan& p = sb.plan;
  char buf[1024];
  std::snprintf(buf, sizeof(buf),
                "{\"kernel\":\"sab\",\"ncol\":%u,\"ta\":%u,\"rpt\":%d,\"n_tiles\":%u,"
                "\"n_beta\":%u,\"grid\":%u,\"slots_a\":%u,\"slots_b\":%u,\"n_a\":%llu,"
                "\"n_b\":%llu,\"ws_bytes\":%zu,\"smem\":%u,\"outer_dims\":%d,\"inner_dims\":%d,"
                "\"beta_dims\":%d,\"ring\":%u}",
                p.ncol, p.ta, sb.rpt, p.n_tiles, p.n_beta, p.grid, p.slots_a, p.n_tiles,
                (unsigned long long)p.n_a, (unsigned long long)p.n_b,
                sb.ws_a_bytes + sb.ws_b_bytes, p.smem_bytes, p.a_outer.n, p.a_inner.n, p.beta.n, p.ring);
  return buf;
}

}  // namespace zr
