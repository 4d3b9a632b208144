// zr_internal.h — plan structures shared by the host planner and the CUDA
// kernels.  Everything here is plain data passed to kernels by value (the
// "DimsArg" idea of the Zero book's GPU page, section Kernel 派发: up to eight
// dimensions travel as kernel parameters, with no metadata copies), plus the
// integer fast-divmod used to turn a linear index into coordinates, and the
// block/item index maps that both the kernels and the host-side plan checker
// use.
#pragma once

#include <stdint.h>
#include <stddef.h>

#if defined(__CUDACC__)
#define ZR_HD __host__ __device__ __forceinline__
#define ZR_CX __host__ __device__ constexpr
#else
#define ZR_HD inline
#define ZR_CX constexpr
#endif

namespace zr {

constexpr int kMaxDims = 8;
// Operand slots of a plan.  Slots 0..2 are inputs, slot 3 the output offset.
// Forward: A, B, -, OUT.  Backward: G (grad_out), A, B, D (a gradient that
// has the output's shape, written densely).
constexpr int kMaxOperands = 4;
constexpr int kSlotOut = 3;

enum OpCode : int32_t { OP_ADD = 0, OP_SUB = 1, OP_MUL = 2, OP_DIV = 3 };
enum UnaryCode : int32_t { UN_SCALE = 0, UN_GELU = 1 };

// ---------------------------------------------------------------------------
// Division by an invariant unsigned 32-bit integer with one multiply-high,
// one add and one shift (T. Granlund and P. L. Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, section 4): with
// l = ceil(log2 d) and m = floor(2^32 * (2^l - d) / d) + 1,
// floor(n / d) = (mulhi(m, n) + n) >> l for every 0 <= n < 2^32.  The sum is
// formed in 64 bits, so no overflow correction is needed, and d = 1 works
// with l = 0, m = 1 (mulhi gives 0).
struct FastDiv {
  uint32_t d;  // divisor, >= 1
  uint32_t m;  // magic multiplier
  uint32_t l;  // shift
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d == 0 ? 1 : d;
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < f.d) ++l;
  f.l = l;
  // (2^l - d) < d <= 2^32, so the product fits in 64 bits and m < 2^32.
  const uint64_t two32 = uint64_t(1) << 32;
  f.m = static_cast<uint32_t>((two32 * ((uint64_t(1) << l) - f.d)) / f.d + 1);
  return f;
}

ZR_HD uint32_t fd_div(const FastDiv& f, uint32_t n) {
#if defined(__CUDA_ARCH__)
  const uint32_t t = __umulhi(n, f.m);
#else
  const uint32_t t = static_cast<uint32_t>((uint64_t(n) * f.m) >> 32);
#endif
  return static_cast<uint32_t>((uint64_t(t) + n) >> f.l);
}

// Decomposition of a row-major linear index over up to eight dimensions,
// innermost first, accumulating per-operand element offsets.
struct Decomp {
  int32_t n;                                  // number of dims (0 = none)
  FastDiv div[kMaxDims];                      // sizes, innermost first
  int64_t stride[kMaxOperands][kMaxDims];     // per operand, innermost first
};

ZR_HD void decomp_offsets(const Decomp& dc, uint32_t idx, int64_t* off) {
  for (int k = 0; k < kMaxOperands; ++k) off[k] = 0;
  for (int i = 0; i < dc.n; ++i) {
    const uint32_t q = fd_div(dc.div[i], idx);
    const uint32_t c = idx - q * dc.div[i].d;
    idx = q;
#if defined(__CUDA_ARCH__)
#pragma unroll
#endif
    for (int k = 0; k < kMaxOperands; ++k) off[k] += int64_t(c) * dc.stride[k][i];
  }
}

// ---------------------------------------------------------------------------
// Elementwise tile plan (forward; backward when no gradient is reduced;
// sum-to-shape without reduction).  The coalesced output is viewed as
// rows x columns: columns = the innermost coalesced dim (ncol), rows = all
// outer dims (nrow, row-major).  A CTA covers tile_rows consecutive rows and
// tile_vcols vectors of VEC columns; a per-CTA table in shared memory holds
// each row's operand offsets, so index decomposition runs once per row, not
// once per element.
struct EwPlan {
  const float* in[3];       // forward: a, b; backward: g, a, b
  float* out[2];            // forward: out; backward: grad_a, grad_b
  Decomp rows;              // decomposition of the row index (outer dims)
  int64_t inner_stride[kMaxOperands];
  uint32_t stream_mask;     // bit k: input k is full-size (read once)
  uint32_t nrow;            // number of rows
  uint32_t ncol;            // columns per row
  uint32_t nvcol;           // column vectors per row = ceil(ncol / VEC)
  uint32_t tile_rows;       // rows per CTA tile (<= kMaxTileRows)
  uint32_t tile_vcols;      // column vectors per CTA tile
  uint32_t col_tiles;       // tiles along a row
  FastDiv col_tiles_div;    // blockIdx -> (row tile, column tile)
  FastDiv tile_vcols_div;   // item -> (row in tile, column vector)
  uint32_t items_per_cta;   // tile_rows * tile_vcols (flat: items per CTA)
  uint32_t n_cta;
  float alpha;              // the unary ops' scalar (scale's factor)
  // Flat plans (at most one outer dim): item i of the nrow x nvcol grid is
  // row i / nvcol, column vector i % nvcol, and each operand's offset is
  // row * rows.stride[k][0] + column * inner_stride[k], computed per item
  // with no offset table; CTA c takes items [c * items_per_cta,
  // (c + 1) * items_per_cta), a whole number of the kernel's load batches.
  uint32_t flat;
  uint32_t nitems;          // nrow * nvcol (flat plans)
  FastDiv nvcol_div;        // item -> (row, column vector) (flat plans)
};

// Forward with one input read transposed: that input (X) walks the output's
// innermost dim q with a large stride but has unit stride along another dim
// p.  A CTA moves a 32 x 32 (p, q) tile of X through shared memory so that
// X is read along p and the output written along q, both coalesced.
struct TrPlan {
  const float* x;           // the transposed input
  const float* y;           // the other input
  float* out;
  uint32_t x_is_a;          // 1: out = x op y; 0: out = y op x
  Decomp batch;             // all dims but p and q; slots 0: x, 1: y, 3: out
  int64_t xs_q;             // x stride along q (x stride along p is 1)
  int64_t ys_p, ys_q;       // y strides
  int64_t os_p;             // out stride along p (out stride along q is 1)
  uint32_t np, nq;          // sizes of p and q
  uint32_t n_pt, n_qt;      // tiles along p and q
  FastDiv n_qt_div, n_pt_div;
  uint32_t n_cta;
  uint32_t vec_ok;          // x's rows (along p) and out's rows (along q) start
                            // 16-byte aligned: 16-byte loads and stores
};
constexpr uint32_t kTrTile = 32;   // tile extent along q
constexpr uint32_t kTrP = 128;     // tile extent along p

constexpr uint32_t kMaxTileRows = 512;
constexpr int kThreads = 256;
constexpr uint32_t kSms = 152;  // SMs of a GB300
// Resident CTAs per SM the planner sizes grids for (whole waves of
// kSms * occupancy CTAs); each kernel's __launch_bounds__ asks for at least
// this many, and a GPU test checks the runtime's occupancy against them.
constexpr int kOccEwFwd = 4;      // k_elementwise: forward
constexpr int kOccEwBwd = 3;      // k_elementwise: backward without reduction
constexpr int kOccEwCopy = 5;     // k_elementwise: copy (sum-to-shape onto the same shape)
constexpr int kOccGeluFwd = 5;     // GeLU forward, float
constexpr int kOccGeluFwdWide = 6; // GeLU forward, 8-wide bfloat16 (2 items per batch)
// GeLU on bfloat16 storage by table (k_gelu_bf16): one CTA of 1024 threads
// per SM, items per pass 3 (forward) or 2 (backward, two operands) with the
// next pass's loads in flight (the most that fit in 64 registers without
// spilling), taken for flat plans of at least 32,768 elements per SM, where
// each CTA's fill of its table is small beside its share of the stream (on a
// [2048, 3072] activation the table took the forward from 12.3 to 10.2 us;
// at [1024, 3072] both paths took 8.4-8.6 us, below that the arithmetic
// kernel was faster).
constexpr int kGeluTabThreads = 1024;
constexpr int kGeluTabUnrollFwd = 3;
constexpr int kGeluTabUnrollBwd = 2;
constexpr uint64_t kGeluTabMinElems = uint64_t(kSms) << 15;
constexpr int kOccRedAddSub = 4;  // k_reduce: add, sub, sum-to-shape
constexpr int kOccRedMulDiv = 3;  // k_reduce: mul, div
// k_reduce, cluster variant (no second pass): loads per item are 1 for add,
// sub and sum-to-shape, 2 for mul and div (the reduced gradient's own input
// is loaded once per thread, the other one per item).  Items in flight per
// thread: 4 (8 measured slower on c5a's backward, 26.7 against 22.8 us: it
// spilled at the 64-register budget of 4 CTAs per SM).  Inner-reduced plans
// with one load per item keep 4 CTAs per SM, the others 3.
ZR_CX int red_cl_loads(int op) { return (op == OP_MUL || op == OP_DIV) ? 2 : 1; }
ZR_CX int red_cl_unroll(int) { return 4; }
ZR_CX int red_cl_occ(int op, bool inner_kept) {
  return (!inner_kept && red_cl_loads(op) == 1) ? 4 : 3;
}
// CTAs per SM of the 8-wide bfloat16 instantiations where a vector of 8
// values needs more registers than the float kernel's budget (measured
// spills): by default one fewer, or two from 3.  The reduction keeps 4 for
// add/sub (with the inner dim kept, 8 bytes of spill cost less than the
// memory parallelism a fourth CTA adds: c4 in bf16, backward add, 88 against
// 79 us), 3 for mul/div with the inner dim reduced, 2 for mul/div with it
// kept.
ZR_CX int wide_occ(int occ) { return occ >= 4 ? 3 : 2; }
ZR_CX int red_wide_occ(int op, bool inner_kept) {
  return (op == OP_MUL || op == OP_DIV) ? (inner_kept ? 2 : 3) : 4;
}
constexpr uint32_t kMaxCluster = 8;   // CTAs per cluster (the portable limit)
// CTAs of a cluster plan that can be resident at once, out of a full wave of
// `wave` CTAs: clusters must fit within one GPC, which strands slots as the
// cluster grows (measured on GB300 at 3 and 4 CTAs per SM: pairs keep the
// whole wave, up to 4 CTAs about 15/16 of it, up to 8 about 7/8).
ZR_CX uint64_t cluster_wave(uint64_t wave, uint64_t c) {
  return c <= 2 ? wave : (c <= 4 ? wave * 15 / 16 : wave * 7 / 8);
}
constexpr int kOccSabf = 3;       // k_sabf
constexpr int kOccTr = 4;         // k_transpose
// k_transpose: 8 warps x 16 p rows, 8 lanes x 4 q columns.
static_assert(kTrP == (kThreads / 32) * 16 && kTrTile == 32, "transpose tile");

// CTA -> (first row, first column vector, rows in tile, vectors in tile).
struct EwTile {
  uint32_t row0, vcol0, nrows, nvcols;
};
ZR_HD EwTile ew_tile(const EwPlan& p, uint32_t cta) {
  EwTile t;
  const uint32_t rt = fd_div(p.col_tiles_div, cta);
  const uint32_t ct = cta - rt * p.col_tiles;
  t.row0 = rt * p.tile_rows;
  t.vcol0 = ct * p.tile_vcols;
  const uint32_t rleft = p.nrow - t.row0;
  const uint32_t vleft = p.nvcol - t.vcol0;
  t.nrows = rleft < p.tile_rows ? rleft : p.tile_rows;
  t.nvcols = vleft < p.tile_vcols ? vleft : p.tile_vcols;
  return t;
}

// ---------------------------------------------------------------------------
// Reduction plan: one gradient X (or the output of sum-to-shape) that sums
// terms over its broadcast dims, optionally writing one dense gradient D in
// the same pass.  Outer dims split into kept dims K' (X has them) and
// reduced dims R'.  The innermost dim is either kept by X (threads own
// columns and add rows) or reduced (all threads of a CTA add into one value
// per kept index).  Each CTA writes one partial per output it touches, to a
// fixed slot; a second pass adds the slots in order.  No atomics anywhere.
struct RedPlan {
  const float* g;           // grad_out (or sum-to-shape input)
  const float* a;
  const float* b;
  float* x_final;           // X, dense in its own shape (when nslots == 1)
  float* partial;           // workspace partials [nslots][nout] (nslots > 1)
  float* d_out;             // dense gradient written in the same pass, or null
  Decomp kept;              // kept outer dims; operands G, A, B, D
  Decomp red;               // reduced outer dims; operands G, A, B, D
  int64_t inner_stride[kMaxOperands];  // G, A, B, D strides along the inner dim
  uint32_t stream_mask;     // bit k: input k is full-size (read once)
  uint32_t n_kept;          // product of kept outer sizes
  uint32_t n_red;           // product of reduced outer sizes (rows)
  uint32_t ncol;            // inner dim size
  uint32_t nvcol;           // ceil(ncol / VEC)
  uint32_t inner_kept;      // 1: inner dim kept by X; 0: reduced
  uint32_t tx, ty;          // thread layout: tx column lanes x ty row lanes
  uint32_t rows_per_blk;    // rows of the reduced range per CTA (<= kMaxTileRows)
  uint32_t vcols_per_blk;   // column vectors per CTA (multiple of tx)
  uint32_t n_rblk;          // row blocks
  uint32_t n_cblk;          // column blocks
  FastDiv n_cblk_div;
  FastDiv n_rblk_div;
  uint64_t nout;            // elements of X
  uint32_t nslots;          // partial slots per output (1 = final write)
  uint32_t n_cta;
  float scale;              // multiplies X's final value (1 except as noted)
  // Cluster plans (cluster > 1): the CTAs that cover one output tile run as
  // one thread-block cluster of `cluster` CTAs, and the cluster's rank-0 CTA
  // adds their results in rank order from distributed shared memory, so
  // there are no partial slots and no second pass.  Inner dim kept: a tile is
  // (kept index, column block), rank = row block.  Inner dim reduced: a tile
  // is a kept index, rank = row block * n_cblk + column block.
  uint32_t cluster;
  FastDiv cluster_div;
  // cp.async staging of the streamed inputs (16-byte vectors with unit inner
  // stride): a ring of `stages` batches (0 = loads into registers), each
  // holding stage_ns streams x 4 items x 256 threads of 16 bytes, after the
  // offset table and the tree in dynamic shared memory.
  uint32_t stages;
  uint32_t stage_ns;
};
// Bytes of one staged batch per streamed input (4 items x 256 threads x 16).
constexpr uint32_t kStageBatchBytes = 4 * kThreads * 16;
// Shared memory the planner lets one SM's resident CTAs use in total, and
// what each CTA keeps back beyond its own request.
constexpr uint32_t kSmemPerSm = 228 * 1024;
constexpr uint32_t kSmemReservedPerCta = 1024;

struct RedCta {
  uint32_t kidx, rblk, cblk;
};
// CTA order: column blocks fastest, then row blocks, then kept index; in a
// cluster plan, cluster rank fastest, then tile.
ZR_HD RedCta red_cta(const RedPlan& p, uint32_t cta) {
  RedCta c;
  if (p.cluster > 1) {
    const uint32_t tile = fd_div(p.cluster_div, cta);
    const uint32_t rank = cta - tile * p.cluster;
    if (p.inner_kept) {
      c.rblk = rank;
      c.kidx = fd_div(p.n_cblk_div, tile);
      c.cblk = tile - c.kidx * p.n_cblk;
    } else {
      c.kidx = tile;
      c.rblk = fd_div(p.n_cblk_div, rank);
      c.cblk = rank - c.rblk * p.n_cblk;
    }
    return c;
  }
  const uint32_t t = fd_div(p.n_cblk_div, cta);
  c.cblk = cta - t * p.n_cblk;
  c.kidx = fd_div(p.n_rblk_div, t);
  c.rblk = t - c.kidx * p.n_rblk;
  return c;
}

// ---------------------------------------------------------------------------
// Fused backward when BOTH gradients are reduced and the innermost dim is
// kept by both (every other dim is kept by exactly one input).  Writing
// A = the dims only a keeps and B = the dims only b keeps, grad_out is a
// family of matrices g[alpha, beta, col]: grad_a = sum over beta, grad_b =
// sum over alpha.  alpha = (A-outer tile, A-inner row), beta = all B dims.
// A persistent grid of `grid` CTAs splits the step sequence
// (tile, beta), tile-major, into equal contiguous ranges; each step streams
// one tile of ta rows x ncol columns through a shared-memory pipeline.
// grad_a partials are flushed when a CTA leaves a tile (slot = the CTA's
// position among the CTAs covering that tile); grad_b partials are written
// per step (slot = tile).  A second pass adds the slots in order.
struct SabPlan {
  const float* g;
  const float* a;
  const float* b;
  float* ws_a;              // [slots_a][n_a]
  float* ws_b;              // [n_tiles][n_b]
  Decomp a_outer;           // tile -> offsets (slot 0: g, slot 1: a)
  Decomp a_inner;           // row  -> offsets (slot 0: g, slot 1: a)
  Decomp beta;              // beta -> offsets (slot 0: g, slot 2: b)
  uint32_t ncol, nvc;       // inner dim, its float4 count (power of two <= 32)
  uint32_t ta;              // rows per tile
  uint32_t n_tiles, n_beta;
  FastDiv n_beta_div;
  uint64_t total_steps;     // n_tiles * n_beta
  uint32_t grid;            // CTAs (persistent)
  uint32_t slots_a;         // grad_a partial slots (max CTAs covering a tile)
  uint64_t n_a, n_b;        // elements of grad_a / grad_b
  uint32_t ring;            // steps whose grad_b partials wait in shared memory
                            // before one pass sums them (power of two,
                            // ring * ncol <= kSabThreads)
  uint32_t smem_bytes;
};

// Forward for the same split (every outer dim varies in exactly one input,
// the innermost in both): out[alpha, beta, col] = a[alpha, col] op
// b[beta, col].  A CTA holds one tile of a's rows in registers and writes
// them against a chunk of betas, one b row per step.
struct SabFPlan {
  const float* a;
  const float* b;
  float* out;
  Decomp a_outer;           // tile -> offsets (slot 0: out, 1: a)
  Decomp a_inner;           // row  -> offsets (slot 0: out, 1: a)
  Decomp beta;              // beta -> offsets (slot 0: out, 2: b)
  uint32_t ncol, nvc;       // inner dim, float4 count (power of two <= 32)
  uint32_t ta;              // rows per tile
  uint32_t n_tiles, n_beta;
  uint32_t beta_chunk, n_bc;  // betas per CTA, chunks
  FastDiv n_bc_div;
  uint32_t n_cta;
};

constexpr int kSabStages = 5;
constexpr int kSabFold = 8;   // steps summed plainly before a Kahan fold
constexpr int kSabThreads = 512;
constexpr uint32_t kSabGrid = 152;  // one CTA per SM of a GB300; fixed so that
                                    // the partition depends on the shape only

// First step of CTA c, and the CTA that owns a step.
ZR_HD uint64_t sab_start(const SabPlan& p, uint32_t c) {
  return (uint64_t(c) * p.total_steps) / p.grid;
}
ZR_HD uint32_t sab_owner(const SabPlan& p, uint64_t step) {
  return static_cast<uint32_t>(((step + 1) * p.grid - 1) / p.total_steps);
}

// Fused backward of a two-op chain out = (a op1 b) op2 c in one pass over
// grad_out, when a has the output's shape and b is reduced: grad_a is the
// dense gradient (r.d_out), grad_b the reduced one (r's X, inner dim kept,
// 16-byte vectors), and grad_c is summed in the same pass.  Either c has b's
// shape and both are dense, so c's offsets are b's and grad_c shares grad_b's
// tiling and slots (c_scalar = 0): the partials are r.partial[nslots][2 nout],
// grad_b's in the first nout of each slot row and grad_c's in the second, so
// one second pass finishes both.  Or c has one element and grad_c is the total
// sum, one partial per CTA in c_partial[n_cta] (c_scalar = 1).
struct ChainPlan {
  RedPlan r;                // g, a, b, grad_b (x_final / partial), grad_a (d_out)
  const float* c;
  float* c_final;           // grad_c
  float* c_partial;         // c_scalar: grad_c's per-CTA partials
  uint32_t c_scalar;
};
constexpr int kOccChain = 3;  // k_chain_bwd: CTAs per SM

// Second pass: out[j] = sum over s of partial[s * nout + j], s in order.
struct CombinePlan {
  const float* partial;
  float* out;               // outputs j < split
  float* out2;              // outputs j >= split, at out2[j - split]
  uint64_t split;           // nout when every output goes to out
  uint64_t nout;
  uint32_t nslots;
  uint32_t jx, sy;          // thread layout: jx output groups x sy slot lanes
  float scale;
  uint32_t vec;             // outputs per group (1, or 4 with 16-byte partial loads)
  // post = 1: output j's total is multiplied by partial[nslots * nout + j],
  // a factor the first pass stored after the slots (division's -1/b^2,
  // applied once to the whole sum so that no partial can overflow on its
  // own).
  uint32_t post;
};

}  // namespace zr
