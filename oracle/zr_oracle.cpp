// zr_oracle.cpp — plain, slow, obviously correct CPU oracle for broadcasting
// elementwise binary ops (add/sub/mul/div on strided fp32 tensors), their
// backward, and sum-to-shape.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
// calls this file; it shares no code, header, table or helper with the CUDA
// path. Only the tests, the smoke check and the benchmark's CPU-baseline leg
// use it.
//
// Source of the semantics ("Zero" book, ismantic.github.io/zero):
//   * Tensor page, section "形状与步长" (shape and strides): an element at
//     coordinate (i, j, ...) lives at sum_d coord_d * stride_d elements from
//     the base; default row-major strides are built from the last dimension.
//   * Operator page, section "广播" (broadcasting): dims are compared from the
//     last one backwards; each pair must be equal, or one side is 1, or one
//     side is missing (treated as 1); a size-1 input dim always reads
//     coordinate 0.  Repetition in the forward pass means summation in the
//     backward pass: dL/dx_j = sum over every output i that maps to j.
//   * Operator page, section "逐元素算子" (elementwise ops): add, sub, mul,
//     div; for mul, dL/dx = g*y and dL/dy = g*x.
//   * GPU page, section "OpAdd": add's local derivative is 1 for both inputs.
//   * sub and div backward are not written out on the pages; this file uses
//     the calculus rules: sub -> (g, -g); div -> (g/b, -g*a/b^2).
//
// Arithmetic: forward results are one IEEE binary32 operation per element
// (round to nearest even; build with -ffp-contract=off, no fast-math).
// Every gradient is accumulated in binary64 and rounded once to binary32.
// A gradient element that receives exactly one term takes that term's
// binary64 value rounded once; for one +, -, * or / of binary32 operands the
// binary64 result rounded to binary32 equals the direct binary32 operation
// (double rounding is innocuous when the wide format has >= 2p+2 bits:
// 53 >= 2*24+2; S. A. Figueroa, "When is double rounding innocuous?",
// SIGNUM Newsletter 30(3), 1995).  The one multi-op term, -g*a/b^2, is
// computed in binary64.
//
// All functions return 0 on success and a negative code on bad arguments:
//   -2 rank out of range (ndim < 0 or > 8), -3 shapes not broadcastable,
//   -4 negative size or stride, -1 NULL pointer where data is required.

#include <cstdint>
#include <cstddef>
#include <cmath>
#include <cstring>
#include <vector>

namespace {

constexpr int kMaxDims = 8;

enum Op { OP_ADD = 0, OP_SUB = 1, OP_MUL = 2, OP_DIV = 3 };

struct View {
  const float* data;
  int ndim;
  std::vector<int64_t> sizes;
  std::vector<int64_t> strides;  // in elements
};

// Row-major strides computed from the last dimension (Tensor page,
// "形状与步长": [2,3,4] -> [12,4,1]).
std::vector<int64_t> row_major_strides(const std::vector<int64_t>& sizes) {
  std::vector<int64_t> st(sizes.size());
  int64_t s = 1;
  for (int d = static_cast<int>(sizes.size()) - 1; d >= 0; --d) {
    st[d] = s;
    s *= sizes[d];
  }
  return st;
}

int make_view(const float* data, int ndim, const int64_t* sizes,
              const int64_t* strides, View* v) {
  if (ndim < 0 || ndim > kMaxDims) return -2;
  if (ndim > 0 && sizes == nullptr) return -1;
  v->data = data;
  v->ndim = ndim;
  v->sizes.assign(sizes, sizes + ndim);
  for (int d = 0; d < ndim; ++d)
    if (v->sizes[d] < 0) return -4;
  if (strides == nullptr) {
    v->strides = row_major_strides(v->sizes);
  } else {
    v->strides.assign(strides, strides + ndim);
    for (int d = 0; d < ndim; ++d)
      if (v->strides[d] < 0) return -4;
  }
  return 0;
}

int64_t numel(const std::vector<int64_t>& sizes) {
  int64_t n = 1;
  for (int64_t s : sizes) n *= s;
  return n;
}

// Operator page, "广播": compare from the last dim; equal, or one is 1, or
// one is missing.  A size-0 dim pairs with 0 or 1 (the pages are silent on
// empty tensors; this is the NumPy reading).
int broadcast(const std::vector<int64_t>& a, const std::vector<int64_t>& b,
              std::vector<int64_t>* out) {
  const int na = static_cast<int>(a.size());
  const int nb = static_cast<int>(b.size());
  const int n = na > nb ? na : nb;
  out->assign(n, 1);
  for (int k = 0; k < n; ++k) {  // k counts from the last dimension
    const int64_t sa = (k < na) ? a[na - 1 - k] : 1;
    const int64_t sb = (k < nb) ? b[nb - 1 - k] : 1;
    int64_t so;
    if (sa == sb) so = sa;
    else if (sa == 1) so = sb;
    else if (sb == 1) so = sa;
    else return -3;
    (*out)[n - 1 - k] = so;
  }
  return 0;
}

// Element offset of an input for a given output coordinate: the input is
// right-aligned against the output; on a size-1 input dim the coordinate is
// always 0 (Operator page, "广播").
int64_t input_offset(const View& v, const std::vector<int64_t>& out_coord) {
  const int n = static_cast<int>(out_coord.size());
  int64_t off = 0;
  for (int d = 0; d < v.ndim; ++d) {
    const int od = n - v.ndim + d;
    const int64_t c = (v.sizes[d] == 1) ? 0 : out_coord[od];
    off += c * v.strides[d];
  }
  return off;
}

// Linear index, in the input's own dense row-major layout, of the element
// an output coordinate maps to.  This is where that element's gradient goes.
int64_t input_dense_index(const View& v, const std::vector<int64_t>& out_coord) {
  const int n = static_cast<int>(out_coord.size());
  int64_t idx = 0;
  for (int d = 0; d < v.ndim; ++d) {
    const int od = n - v.ndim + d;
    const int64_t c = (v.sizes[d] == 1) ? 0 : out_coord[od];
    idx = idx * v.sizes[d] + c;
  }
  return idx;
}

// Odometer step over a shape, last dim fastest (row-major order).
bool next_coord(std::vector<int64_t>* c, const std::vector<int64_t>& sizes) {
  for (int d = static_cast<int>(sizes.size()) - 1; d >= 0; --d) {
    if (++(*c)[d] < sizes[d]) return true;
    (*c)[d] = 0;
  }
  return false;
}

std::vector<int64_t> unravel(int64_t i, const std::vector<int64_t>& sizes) {
  std::vector<int64_t> c(sizes.size(), 0);
  for (int d = static_cast<int>(sizes.size()) - 1; d >= 0; --d) {
    c[d] = i % sizes[d];
    i /= sizes[d];
  }
  return c;
}

float fwd_op(int op, float x, float y) {
  switch (op) {
    case OP_ADD: return x + y;
    case OP_SUB: return x - y;
    case OP_MUL: return x * y;
    default:     return x / y;
  }
}

// Local gradient terms in binary64 from binary32 inputs.
//   add: (g, g)            GPU page, "OpAdd"
//   sub: (g, -g)           calculus
//   mul: (g*y, g*x)        Operator page, "逐元素算子"
//   div: (g/y, -g*x/y^2)   calculus
double term_a(int op, double g, double x, double y) {
  (void)x;
  switch (op) {
    case OP_ADD: return g;
    case OP_SUB: return g;
    case OP_MUL: return g * y;
    default:     return g / y;
  }
}
double term_b(int op, double g, double x, double y) {
  switch (op) {
    case OP_ADD: return g;
    case OP_SUB: return -g;
    case OP_MUL: return g * x;
    default:     return -(g * x) / (y * y);
  }
}

bool op_needs_a(int op, int which) {  // which: 0 -> grad_a, 1 -> grad_b
  if (op == OP_MUL) return which == 1;
  if (op == OP_DIV) return which == 1;
  return false;
}
bool op_needs_b(int op, int which) {
  if (op == OP_MUL) return which == 0;
  if (op == OP_DIV) return true;
  return false;
}

}  // namespace

extern "C" {

// Default row-major strides of a shape (Tensor page, "形状与步长").
int orc_contiguous_strides(int ndim, const int64_t* sizes, int64_t* strides) {
  if (ndim < 0 || ndim > kMaxDims) return -2;
  std::vector<int64_t> s(sizes, sizes + ndim);
  std::vector<int64_t> st = row_major_strides(s);
  for (int d = 0; d < ndim; ++d) strides[d] = st[d];
  return 0;
}

// Broadcast shape of two shapes (Operator page, "广播").
int orc_broadcast_shape(int ndim_a, const int64_t* sizes_a, int ndim_b,
                        const int64_t* sizes_b, int* ndim_out,
                        int64_t* sizes_out) {
  if (ndim_a < 0 || ndim_a > kMaxDims || ndim_b < 0 || ndim_b > kMaxDims)
    return -2;
  std::vector<int64_t> a(sizes_a, sizes_a + ndim_a);
  std::vector<int64_t> b(sizes_b, sizes_b + ndim_b);
  for (int64_t s : a) if (s < 0) return -4;
  for (int64_t s : b) if (s < 0) return -4;
  std::vector<int64_t> o;
  const int rc = broadcast(a, b, &o);
  if (rc) return rc;
  *ndim_out = static_cast<int>(o.size());
  for (size_t d = 0; d < o.size(); ++d) sizes_out[d] = o[d];
  return 0;
}

// Forward: out (dense row-major, broadcast shape) = a op b, one binary32 op
// per element, inputs read through their strides.
int orc_binary_fwd(int op,
                   const float* a, int nda, const int64_t* sza, const int64_t* sta,
                   const float* b, int ndb, const int64_t* szb, const int64_t* stb,
                   float* out) {
  if (op < 0 || op > 3) return -1;
  View va, vb;
  int rc = make_view(a, nda, sza, sta, &va);
  if (rc) return rc;
  rc = make_view(b, ndb, szb, stb, &vb);
  if (rc) return rc;
  std::vector<int64_t> os;
  rc = broadcast(va.sizes, vb.sizes, &os);
  if (rc) return rc;
  const int64_t n = numel(os);
  if (n == 0) return 0;
  if (!a || !b || !out) return -1;
  std::vector<int64_t> c(os.size(), 0);
  int64_t i = 0;
  do {
    out[i++] = fwd_op(op, a[input_offset(va, c)], b[input_offset(vb, c)]);
  } while (next_coord(&c, os));
  return 0;
}

// Forward at selected output linear indices (row-major in the broadcast
// shape): vals[k] = out[idx[k]].  Same arithmetic as orc_binary_fwd.
int orc_binary_fwd_at(int op,
                      const float* a, int nda, const int64_t* sza, const int64_t* sta,
                      const float* b, int ndb, const int64_t* szb, const int64_t* stb,
                      int64_t n_idx, const int64_t* idx, float* vals) {
  if (op < 0 || op > 3) return -1;
  View va, vb;
  int rc = make_view(a, nda, sza, sta, &va);
  if (rc) return rc;
  rc = make_view(b, ndb, szb, stb, &vb);
  if (rc) return rc;
  std::vector<int64_t> os;
  rc = broadcast(va.sizes, vb.sizes, &os);
  if (rc) return rc;
  const int64_t n = numel(os);
  for (int64_t k = 0; k < n_idx; ++k) {
    if (idx[k] < 0 || idx[k] >= n) return -4;
    const std::vector<int64_t> c = unravel(idx[k], os);
    vals[k] = fwd_op(op, a[input_offset(va, c)], b[input_offset(vb, c)]);
  }
  return 0;
}

// Backward by the definition, scattering: for every output coordinate i
// (row-major order), the local terms of i are added into the gradient
// element that i maps to in each input's own shape.  grad_a / grad_b are
// dense row-major in a's / b's shape and may be NULL (skipped).  abs_a /
// abs_b (nullable) receive sum |term| per gradient element, in binary64.
// g is read through its strides and must have the broadcast shape.  a (b)
// data may be NULL when no requested gradient needs it.
int orc_binary_bwd(int op,
                   const float* g, int ndg, const int64_t* szg, const int64_t* stg,
                   const float* a, int nda, const int64_t* sza, const int64_t* sta,
                   const float* b, int ndb, const int64_t* szb, const int64_t* stb,
                   float* grad_a, float* grad_b, double* abs_a, double* abs_b) {
  if (op < 0 || op > 3) return -1;
  View vg, va, vb;
  int rc = make_view(g, ndg, szg, stg, &vg);
  if (rc) return rc;
  rc = make_view(a, nda, sza, sta, &va);
  if (rc) return rc;
  rc = make_view(b, ndb, szb, stb, &vb);
  if (rc) return rc;
  std::vector<int64_t> os;
  rc = broadcast(va.sizes, vb.sizes, &os);
  if (rc) return rc;
  if (vg.sizes != os) return -3;
  const bool want_a = grad_a != nullptr;
  const bool want_b = grad_b != nullptr;
  const bool need_a = (want_a && op_needs_a(op, 0)) || (want_b && op_needs_a(op, 1));
  const bool need_b = (want_a && op_needs_b(op, 0)) || (want_b && op_needs_b(op, 1));
  const int64_t n = numel(os);
  const int64_t na = numel(va.sizes), nb = numel(vb.sizes);
  std::vector<double> acc_a(want_a ? na : 0, 0.0), acc_b(want_b ? nb : 0, 0.0);
  std::vector<double> sa(want_a ? na : 0, 0.0), sb(want_b ? nb : 0, 0.0);
  std::vector<unsigned char> seen_a(want_a ? na : 0, 0), seen_b(want_b ? nb : 0, 0);
  if (n > 0) {
    if (!g || (need_a && !a) || (need_b && !b)) return -1;
    std::vector<int64_t> c(os.size(), 0);
    do {
      const double gv = g[input_offset(vg, c)];
      const double av = need_a ? static_cast<double>(a[input_offset(va, c)]) : 0.0;
      const double bv = need_b ? static_cast<double>(b[input_offset(vb, c)]) : 0.0;
      if (want_a) {
        const int64_t j = input_dense_index(va, c);
        const double t = term_a(op, gv, av, bv);
        // The first term is taken as is, so that a gradient element with a
        // single term keeps that term's sign of zero.
        acc_a[j] = seen_a[j] ? acc_a[j] + t : t;
        seen_a[j] = 1;
        sa[j] += std::fabs(t);
      }
      if (want_b) {
        const int64_t j = input_dense_index(vb, c);
        const double t = term_b(op, gv, av, bv);
        acc_b[j] = seen_b[j] ? acc_b[j] + t : t;
        seen_b[j] = 1;
        sb[j] += std::fabs(t);
      }
    } while (next_coord(&c, os));
  }
  // A gradient element that no output maps to (only possible when the
  // output is empty) is 0.
  for (int64_t j = 0; j < (want_a ? na : 0); ++j) {
    grad_a[j] = static_cast<float>(acc_a[j]);
    if (abs_a) abs_a[j] = sa[j];
  }
  for (int64_t j = 0; j < (want_b ? nb : 0); ++j) {
    grad_b[j] = static_cast<float>(acc_b[j]);
    if (abs_b) abs_b[j] = sb[j];
  }
  return 0;
}

// Backward at selected gradient elements, gathering: for each requested
// element j (row-major in the input's shape) of grad_a (which == 0) or grad_b
// (which == 1), enumerate every output coordinate that maps to j in
// row-major order and sum its terms in binary64.  This is the per-output
// form of the same definition and is used where the output is too large to
// enumerate.
int orc_binary_bwd_at(int op, int which,
                      const float* g, int ndg, const int64_t* szg, const int64_t* stg,
                      const float* a, int nda, const int64_t* sza, const int64_t* sta,
                      const float* b, int ndb, const int64_t* szb, const int64_t* stb,
                      int64_t n_idx, const int64_t* idx, float* vals, double* abs_vals) {
  if (op < 0 || op > 3 || which < 0 || which > 1) return -1;
  View vg, va, vb;
  int rc = make_view(g, ndg, szg, stg, &vg);
  if (rc) return rc;
  rc = make_view(a, nda, sza, sta, &va);
  if (rc) return rc;
  rc = make_view(b, ndb, szb, stb, &vb);
  if (rc) return rc;
  std::vector<int64_t> os;
  rc = broadcast(va.sizes, vb.sizes, &os);
  if (rc) return rc;
  if (vg.sizes != os) return -3;
  const bool need_a = op_needs_a(op, which);
  const bool need_b = op_needs_b(op, which);
  const View& vx = which == 0 ? va : vb;
  const int n = static_cast<int>(os.size());
  const int64_t nx = numel(vx.sizes);
  for (int64_t k = 0; k < n_idx; ++k) {
    if (idx[k] < 0 || idx[k] >= nx) return -4;
    // Coordinate of j in x's own shape, right-aligned to the output.
    const std::vector<int64_t> xc = unravel(idx[k], vx.sizes);
    // Free dims: those where x is 1 (or missing) and the output is not.
    std::vector<int64_t> fixed(n, -1), free_sizes;
    std::vector<int> free_dims;
    for (int od = 0; od < n; ++od) {
      const int d = od - (n - vx.ndim);
      if (d >= 0 && vx.sizes[d] != 1) fixed[od] = xc[d];
      else if (os[od] != 1) { free_dims.push_back(od); free_sizes.push_back(os[od]); }
      else fixed[od] = 0;
    }
    double acc = 0.0, sabs = 0.0;
    bool seen = false;
    if (numel(os) > 0) {
      if (!g || (need_a && !a) || (need_b && !b)) return -1;
      std::vector<int64_t> fc(free_sizes.size(), 0);
      std::vector<int64_t> c(n, 0);
      bool more = true;
      while (more) {
        for (int od = 0; od < n; ++od) if (fixed[od] >= 0) c[od] = fixed[od];
        for (size_t f = 0; f < free_dims.size(); ++f) c[free_dims[f]] = fc[f];
        const double gv = g[input_offset(vg, c)];
        const double av = need_a ? static_cast<double>(a[input_offset(va, c)]) : 0.0;
        const double bv = need_b ? static_cast<double>(b[input_offset(vb, c)]) : 0.0;
        const double t = which == 0 ? term_a(op, gv, av, bv) : term_b(op, gv, av, bv);
        acc = seen ? acc + t : t;
        seen = true;
        sabs += std::fabs(t);
        more = !free_sizes.empty() && next_coord(&fc, free_sizes);
      }
    }
    vals[k] = static_cast<float>(acc);
    if (abs_vals) abs_vals[k] = sabs;
  }
  return 0;
}

// Sum-to-shape (Operator page, "广播", OpSumToSize): out (dense row-major,
// shape sizes_out) receives, at each element j, the binary64 sum of every
// input element that maps to j, rounded once.  sizes_out must broadcast
// with the input's shape to exactly the input's shape.  abs_out (nullable)
// receives sum |x| per element.
int orc_sum_to_shape(const float* x, int ndx, const int64_t* szx, const int64_t* stx,
                     int ndo, const int64_t* szo, float* out, double* abs_out) {
  View vx, vo;
  int rc = make_view(x, ndx, szx, stx, &vx);
  if (rc) return rc;
  rc = make_view(nullptr, ndo, szo, nullptr, &vo);
  if (rc) return rc;
  std::vector<int64_t> bs;
  rc = broadcast(vx.sizes, vo.sizes, &bs);
  if (rc) return rc;
  if (bs != vx.sizes) return -3;
  const int64_t n = numel(vx.sizes), no = numel(vo.sizes);
  std::vector<double> acc(no, 0.0), sabs(no, 0.0);
  std::vector<unsigned char> seen(no, 0);
  if (n > 0) {
    if (!x) return -1;
    std::vector<int64_t> c(vx.sizes.size(), 0);
    do {
      const double t = x[input_offset(vx, c)];
      const int64_t j = input_dense_index(vo, c);
      acc[j] = seen[j] ? acc[j] + t : t;
      seen[j] = 1;
      sabs[j] += std::fabs(t);
    } while (next_coord(&c, vx.sizes));
  }
  for (int64_t j = 0; j < no; ++j) {
    out[j] = static_cast<float>(acc[j]);
    if (abs_out) abs_out[j] = sabs[j];
  }
  return 0;
}

// Sum-to-shape at selected output elements (gathering form).
int orc_sum_to_shape_at(const float* x, int ndx, const int64_t* szx, const int64_t* stx,
                        int ndo, const int64_t* szo, int64_t n_idx, const int64_t* idx,
                        float* vals, double* abs_vals) {
  View vx, vo;
  int rc = make_view(x, ndx, szx, stx, &vx);
  if (rc) return rc;
  rc = make_view(nullptr, ndo, szo, nullptr, &vo);
  if (rc) return rc;
  std::vector<int64_t> bs;
  rc = broadcast(vx.sizes, vo.sizes, &bs);
  if (rc) return rc;
  if (bs != vx.sizes) return -3;
  const int n = static_cast<int>(vx.sizes.size());
  const int64_t no = numel(vo.sizes);
  for (int64_t k = 0; k < n_idx; ++k) {
    if (idx[k] < 0 || idx[k] >= no) return -4;
    const std::vector<int64_t> oc = unravel(idx[k], vo.sizes);
    std::vector<int64_t> fixed(n, -1), free_sizes;
    std::vector<int> free_dims;
    for (int xd = 0; xd < n; ++xd) {
      const int d = xd - (n - vo.ndim);
      if (d >= 0 && vo.sizes[d] != 1) fixed[xd] = oc[d];
      else if (vx.sizes[xd] != 1) { free_dims.push_back(xd); free_sizes.push_back(vx.sizes[xd]); }
      else fixed[xd] = 0;
    }
    double acc = 0.0, sabs = 0.0;
    bool seen = false;
    if (numel(vx.sizes) > 0) {
      if (!x) return -1;
      std::vector<int64_t> fc(free_sizes.size(), 0), c(n, 0);
      bool more = true;
      while (more) {
        for (int xd = 0; xd < n; ++xd) if (fixed[xd] >= 0) c[xd] = fixed[xd];
        for (size_t f = 0; f < free_dims.size(); ++f) c[free_dims[f]] = fc[f];
        const double t = x[input_offset(vx, c)];
        acc = seen ? acc + t : t;
        seen = true;
        sabs += std::fabs(t);
        more = !free_sizes.empty() && next_coord(&fc, free_sizes);
      }
    }
    vals[k] = static_cast<float>(acc);
    if (abs_vals) abs_vals[k] = sabs;
  }
  return 0;
}

}  // extern "C"

// ---------------------------------------------------------------- bf16 storage
//
// bfloat16 keeps binary32's sign and 8-bit exponent and the top 7 bits of
// its 23-bit fraction.  Rounding a binary32 value to it, to nearest with
// ties to even: add 0x7FFF plus the lowest kept bit to the bit pattern and
// drop the low 16 bits (a carry into the exponent is the correct rounding up,
// up to infinity); NaN stays NaN (quietened).  Results are returned as the
// binary32 values they denote.
extern "C" int orc_round_bf16(const float* x, int64_t n, float* out) {
  if (n > 0 && (!x || !out)) return -1;
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u;
    std::memcpy(&u, &x[i], 4);
    uint32_t r;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) {
      r = (u | 0x00400000u) & 0xFFFF0000u;
    } else {
      r = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    }
    std::memcpy(&out[i], &r, 4);
  }
  return 0;
}

// ---------------------------------------------------------------- unary ops
//
// GPU page, section 逐元素运算 (elementwise ops): add, mul, GeLU and
// gradient scaling each compute an output element from the input element at
// the same position.  The pages name GeLU without a formula; the plainest
// reading is its exact definition GeLU(x) = x * Phi(x), Phi the standard
// normal CDF, written Phi(x) = erfc(-x / sqrt(2)) / 2.  Evaluated in binary64
// and rounded once.  Backward: d/dx GeLU = Phi(x) + x * phi(x) with
// phi(x) = exp(-x^2 / 2) / sqrt(2 pi).  scale: out = alpha * x, one binary32
// multiply; its backward alpha * g.  Outputs are dense row-major of x's shape.
namespace {
enum Unary { UN_SCALE = 0, UN_GELU = 1 };

double norm_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }
double norm_pdf(double x) { return std::exp(-0.5 * x * x) / std::sqrt(2.0 * 3.14159265358979323846); }

// Visit every element of a strided view in row-major coordinate order.
template <class F>
void for_each_elem(const View& v, F f) {
  const int64_t n = numel(v.sizes);
  std::vector<int64_t> c(v.ndim, 0);
  for (int64_t i = 0; i < n; ++i) {
    int64_t off = 0;
    for (int d = 0; d < v.ndim; ++d) off += c[d] * v.strides[d];
    f(i, off);
    for (int d = v.ndim - 1; d >= 0; --d) {
      if (++c[d] < v.sizes[d]) break;
      c[d] = 0;
    }
  }
}
}  // namespace

extern "C" {

int orc_unary_fwd(int op, float alpha, const float* x, int ndx, const int64_t* szx,
                  const int64_t* stx, float* out) {
  if (op != UN_SCALE && op != UN_GELU) return -1;
  View vx;
  int rc = make_view(x, ndx, szx, stx, &vx);
  if (rc) return rc;
  if (numel(vx.sizes) > 0 && (!x || !out)) return -1;
  for_each_elem(vx, [&](int64_t i, int64_t off) {
    const float xv = x[off];
    if (op == UN_SCALE) {
      out[i] = alpha * xv;
    } else {
      const double xd = xv;
      out[i] = static_cast<float>(xd * norm_cdf(xd));
    }
  });
  return 0;
}

// grad_x[i] = g[i] * f'(x[i]); mag[i] = |g| * (Phi(x) + |x| phi(x)) for GeLU
// (the size of the two terms before they cancel near the minimum at
// x = -0.75), |alpha * g| for scale.
int orc_unary_bwd(int op, float alpha, const float* g, int ndg, const int64_t* szg,
                  const int64_t* stg, const float* x, const int64_t* stx, float* grad_x,
                  double* mag) {
  if (op != UN_SCALE && op != UN_GELU) return -1;
  View vg, vx;
  int rc = make_view(g, ndg, szg, stg, &vg);
  if (rc) return rc;
  rc = make_view(x, ndg, szg, stx, &vx);
  if (rc) return rc;
  const int64_t n = numel(vg.sizes);
  if (n > 0 && (!g || !grad_x || (op == UN_GELU && !x))) return -1;
  std::vector<int64_t> goff(n), xoff(n);
  for_each_elem(vg, [&](int64_t i, int64_t off) { goff[i] = off; });
  for_each_elem(vx, [&](int64_t i, int64_t off) { xoff[i] = off; });
  for (int64_t i = 0; i < n; ++i) {
    const float gv = g[goff[i]];
    if (op == UN_SCALE) {
      grad_x[i] = alpha * gv;
      if (mag) mag[i] = std::fabs(static_cast<double>(alpha) * gv);
    } else {
      const double xd = x[xoff[i]];
      const double cdf = norm_cdf(xd), pdf = norm_pdf(xd);
      grad_x[i] = static_cast<float>(static_cast<double>(gv) * (cdf + xd * pdf));
      if (mag) mag[i] = std::fabs(static_cast<double>(gv)) * (cdf + std::fabs(xd) * pdf);
    }
  }
  return 0;
}

}  // extern "C"
