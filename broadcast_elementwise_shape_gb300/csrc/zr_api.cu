// zr_api.cu — the C ABI (include/zr.h): argument checks, planning and
// launches.  Every check runs on the host before the first launch (Zero book,
// Operator page, section 逐元素算子: shape and broadcast checks belong to the
// operator layer), so an error never leaves a partial write.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/zr.h"
#include "../../include/zr_testing.h"
#include "zr_launch.h"
#include "zr_plan.h"

namespace zr {
namespace {

bool op_ok(int op) { return op >= OP_ADD && op <= OP_DIV; }

// Which inputs a gradient's local term reads (mul: the other input; div:
// b for grad_a, a and b for grad_b).
bool needs_a(int op, int which) { return which == 1 && (op == OP_MUL || op == OP_DIV); }
bool needs_b(int op, int which) {
  return (which == 0 && (op == OP_MUL || op == OP_DIV)) || (which == 1 && op == OP_DIV);
}

// Byte interval [lo, hi) touched by a tensor (empty when numel == 0).
struct Span {
  uintptr_t lo = 0, hi = 0;
};
Span span_of(const void* p, int64_t extent, int es = 4) {
  Span s;
  if (p && extent > 0) {
    s.lo = reinterpret_cast<uintptr_t>(p);
    s.hi = s.lo + uintptr_t(extent) * uintptr_t(es);
  }
  return s;
}
bool overlaps(const Span& x, const Span& y) {
  return x.hi > x.lo && y.hi > y.lo && x.lo < y.hi && y.lo < x.hi;
}

// Sufficient condition for a strided view to address every element once:
// sorted by stride, each stride exceeds the extent of all smaller dims.
bool non_overlapping(const TDesc& t) {
  int idx[kMaxDims];
  int m = 0;
  for (int i = 0; i < t.nd; ++i)
    if (t.size[i] > 1) idx[m++] = i;
  std::sort(idx, idx + m, [&](int x, int y) { return t.stride[x] < t.stride[y]; });
  int64_t reach = 0;  // largest offset reachable with the dims seen so far
  for (int i = 0; i < m; ++i) {
    const int d = idx[i];
    if (t.stride[d] <= reach) return false;
    reach += (t.size[d] - 1) * t.stride[d];
  }
  return true;
}

bool same_layout(const TDesc& x, const TDesc& y) {
  if (x.ptr != y.ptr || x.nd != y.nd) return false;
  for (int i = 0; i < x.nd; ++i) {
    if (x.size[i] != y.size[i]) return false;
    if (x.size[i] > 1 && x.stride[i] != y.stride[i]) return false;
  }
  return true;
}

bool is_reduced(const TDesc& x, int n, const int64_t* out_size) {
  for (int od = 0; od < n; ++od) {
    const int d = od - (n - x.nd);
    if (out_size[od] != 1 && (d < 0 || x.size[d] == 1)) return true;
  }
  return false;
}

TDesc dense_desc(const float* p, int nd, const int64_t* size) {
  TDesc t;
  t.ptr = p;
  t.nd = nd;
  int64_t n = 1;
  for (int i = 0; i < nd; ++i) {
    t.size[i] = size[i];
    n *= size[i];
  }
  t.numel = n;
  contiguous_strides(nd, t.size, t.stride);
  t.extent = n;
  return t;
}

int check_device_ptr(const void* p) {
  if (p == nullptr) return ZR_ERR_NULL;
  cudaPointerAttributes at;
  const cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ZR_ERR_DEVICE;
  }
  if (at.type == cudaMemoryTypeUnregistered) return ZR_ERR_DEVICE;
  // Pinned host memory is used through the same address only (unified
  // addressing maps it there); a different device alias is refused.
  if (at.type == cudaMemoryTypeHost && at.devicePointer != p) return ZR_ERR_DEVICE;
  if (at.type == cudaMemoryTypeDevice) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return ZR_ERR_DEVICE;
    }
    if (at.device != dev) return ZR_ERR_DEVICE;
  }
  return ZR_OK;
}

// ------------------------------------------------------------------ forward

struct FwdSet {
  int es = 4;                    // bytes per stored element: 4 float, 2 bfloat16
  int op = 0;
  bool empty = false;
  bool tr = false;               // transposed-input tile path
  TrPlan tp;
  bool sabf = false;             // split forward path
  SabFPlan sp;
  int sp_rpt = 0;
  EwBuild eb;
  TDesc a, b, out;
};

int plan_fwd(int op, const zr_tensor& ta, const zr_tensor& tb, const float* out,
             const int64_t* out_strides, FwdSet* S) {
  if (!op_ok(op)) return ZR_ERR_NULL;
  S->op = op;
  int rc = read_tensor(ta, &S->a);
  if (rc) return rc;
  rc = read_tensor(tb, &S->b);
  if (rc) return rc;
  int n = 0;
  int64_t osz[kMaxDims];
  rc = broadcast_sizes(S->a.nd, S->a.size, S->b.nd, S->b.size, &n, osz);
  if (rc) return rc;
  zr_tensor to{out, n, osz, out_strides};
  rc = read_tensor(to, &S->out);
  if (rc) return rc;
  if (S->out.numel == 0) {
    S->empty = true;
    return ZR_OK;
  }
  if (!S->a.ptr || !S->b.ptr || !out) return ZR_ERR_NULL;
  if (!non_overlapping(S->out)) return ZR_ERR_LAYOUT;
  const Span so = span_of(out, S->out.extent, S->es);
  for (const TDesc* x : {&S->a, &S->b}) {
    if (overlaps(so, span_of(x->ptr, x->extent, S->es)) && !same_layout(*x, S->out))
      return ZR_ERR_LAYOUT;
  }
  int64_t st[kProbSlots][kMaxDims] = {};
  align_strides(S->a, n, osz, st[0]);
  align_strides(S->b, n, osz, st[1]);
  for (int d = 0; d < n; ++d) st[kSlotOut][d] = osz[d] == 1 ? 0 : S->out.stride[d];
  Prob P;
  rc = coalesce(n, osz, st, (1u << 0) | (1u << 1) | (1u << kSlotOut), kSlotOut, &P);
  if (rc) return rc;
  P.es = S->es;
  const float* in[3] = {S->a.ptr, S->b.ptr, nullptr};
  float* outs[2] = {const_cast<float*>(out), nullptr};
  const uint32_t stream_mask = (S->a.numel == S->out.numel ? 1u : 0u) |
                               (S->b.numel == S->out.numel ? 2u : 0u);
  // The transposed-tile and split kernels are built for float storage only.
  rc = S->es == 4 ? build_tr(P, S->a.ptr, S->b.ptr, const_cast<float*>(out), &S->tp) : 1;
  if (rc == ZR_OK) {
    S->tr = true;
    return ZR_OK;
  }
  rc = S->es == 4 ? build_sabf(P, S->a.ptr, S->b.ptr, const_cast<float*>(out), &S->sp, &S->sp_rpt)
                   : 1;
  if (rc == ZR_OK) {
    S->sabf = true;
    return ZR_OK;
  }
  rc = build_ew(P, in, outs, 0x3u, stream_mask, kOccEwFwd, &S->eb);
  S->eb.uni1 = S->b.numel == 1;
  return rc;
}

// ------------------------------------------------------------------ backward

struct BwdSet {
  int es = 4;                    // bytes per stored element: 4 float, 2 bfloat16
  int op = 0;
  bool nothing = false;          // no gradient requested
  bool empty = false;            // grad_out empty: only zero fills
  bool direct = false;           // elementwise plan (no reduction)
  int want = 0;                  // bit 0 grad_a, bit 1 grad_b
  EwBuild eb;
  int nred = 0;
  int which[2] = {0, 0};
  RedBuild rb[2];
  bool sab = false;              // fused both-reduced pass (k_sab)
  SabBuild sb;
  size_t ws_off[2] = {0, 0};
  size_t ws_run = 0;             // bytes this call uses
  size_t ws_query = 0;           // bytes reported by a workspace query
  float* zero_ptr[2] = {nullptr, nullptr};
  size_t zero_bytes[2] = {0, 0};
  TDesc g, a, b, ga, gb;
};

int plan_bwd(int op, const zr_tensor& tg, const zr_tensor& ta, const zr_tensor& tb, float* grad_a,
             float* grad_b, BwdSet* S) {
  if (!op_ok(op)) return ZR_ERR_NULL;
  S->op = op;
  int rc = read_tensor(tg, &S->g);
  if (rc) return rc;
  rc = read_tensor(ta, &S->a);
  if (rc) return rc;
  rc = read_tensor(tb, &S->b);
  if (rc) return rc;
  int n = 0;
  int64_t osz[kMaxDims];
  rc = broadcast_sizes(S->a.nd, S->a.size, S->b.nd, S->b.size, &n, osz);
  if (rc) return rc;
  if (S->g.nd != n) return ZR_ERR_SHAPE;
  for (int d = 0; d < n; ++d)
    if (S->g.size[d] != osz[d]) return ZR_ERR_SHAPE;
  S->want = (grad_a ? 1 : 0) | (grad_b ? 2 : 0);
  if (S->want == 0) {
    S->nothing = true;
    return ZR_OK;
  }
  S->ga = dense_desc(grad_a, S->a.nd, S->a.size);
  S->gb = dense_desc(grad_b, S->b.nd, S->b.size);
  const bool red_a = grad_a && is_reduced(S->a, n, osz);
  const bool red_b = grad_b && is_reduced(S->b, n, osz);
  const bool read_a = (grad_a && needs_a(op, 0)) || (grad_b && needs_a(op, 1));
  const bool read_b = (grad_a && needs_b(op, 0)) || (grad_b && needs_b(op, 1));

  // Layout: the two gradients are disjoint; a gradient may alias grad_out
  // exactly only when it has grad_out's shape and grad_out is dense (then each
  // element is read and written by the same thread); any other overlap with
  // an input is refused.
  const Span sga = span_of(grad_a, S->ga.extent, S->es);
  const Span sgb = span_of(grad_b, S->gb.extent, S->es);
  if (overlaps(sga, sgb)) return ZR_ERR_LAYOUT;
  struct In { const TDesc* t; bool read; };
  const In ins[3] = {{&S->g, true}, {&S->a, read_a}, {&S->b, read_b}};
  for (int w = 0; w < 2; ++w) {
    const TDesc& gd = w == 0 ? S->ga : S->gb;
    const Span& sp = w == 0 ? sga : sgb;
    const bool reduced = w == 0 ? red_a : red_b;
    if (!gd.ptr) continue;
    for (int i = 0; i < 3; ++i) {
      if (!ins[i].read || !ins[i].t->ptr) continue;
      if (!overlaps(sp, span_of(ins[i].t->ptr, ins[i].t->extent, S->es))) continue;
      const bool ok = i == 0 && !reduced && same_layout(gd, S->g);
      if (!ok) return ZR_ERR_LAYOUT;
    }
  }

  if (S->g.numel == 0) {
    S->empty = true;
    if (grad_a && S->ga.numel > 0) { S->zero_ptr[0] = grad_a; S->zero_bytes[0] = S->ga.numel * S->es; }
    if (grad_b && S->gb.numel > 0) { S->zero_ptr[1] = grad_b; S->zero_bytes[1] = S->gb.numel * S->es; }
    return ZR_OK;
  }
  if (!S->g.ptr || (read_a && !S->a.ptr) || (read_b && !S->b.ptr)) return ZR_ERR_NULL;

  int64_t st[kProbSlots][kMaxDims] = {};
  align_strides(S->g, n, osz, st[0]);
  if (read_a) align_strides(S->a, n, osz, st[1]);
  if (read_b) align_strides(S->b, n, osz, st[2]);
  int64_t dense[kMaxDims];
  contiguous_strides(n, osz, dense);
  for (int d = 0; d < n; ++d) st[kSlotOut][d] = osz[d] == 1 ? 0 : dense[d];
  if (grad_a) grad_index_strides(S->a, n, osz, st[kSlotXA]);
  if (grad_b) grad_index_strides(S->b, n, osz, st[kSlotXB]);
  const uint32_t read_mask = 1u | (read_a ? 2u : 0u) | (read_b ? 4u : 0u);
  const uint32_t stream_mask = 1u | (S->a.numel == S->g.numel ? 2u : 0u) |
                               (S->b.numel == S->g.numel ? 4u : 0u);

  if (!red_a && !red_b) {
    S->direct = true;
    Prob P;
    rc = coalesce(n, osz, st, read_mask | (1u << kSlotOut), -1, &P);
    if (rc) return rc;
    P.es = S->es;
    const float* in[3] = {S->g.ptr, S->a.ptr, S->b.ptr};
    float* outs[2] = {grad_a, grad_b};
    return build_ew(P, in, outs, read_mask, stream_mask, kOccEwBwd, &S->eb);
  }

  // One reduced gradient, the other written densely in the same pass (or
  // not requested); or both reduced, one reduction pass each.
  const bool dense_other = (red_a != red_b) && ((red_a && grad_b) || (red_b && grad_a));
  uint32_t active = read_mask;
  if (dense_other) active |= 1u << kSlotOut;
  if (red_a) active |= 1u << kSlotXA;
  if (red_b) active |= 1u << kSlotXB;
  Prob P;
  rc = coalesce(n, osz, st, active, -1, &P);
  if (rc) return rc;
  P.es = S->es;
  size_t off = 0, off_q = 0;
  for (int w = 0; w < 2; ++w) {
    const bool red = w == 0 ? red_a : red_b;
    if (!red) continue;
    float* xo = w == 0 ? grad_a : grad_b;
    float* d_out = dense_other ? (w == 0 ? grad_b : grad_a) : nullptr;
    const int xslot = w == 0 ? kSlotXA : kSlotXB;
    // Only the operands this gradient's terms need are read in its pass.
    const bool ra = needs_a(op, w) || (d_out && needs_a(op, 1 - w));
    const bool rbb = needs_b(op, w) || (d_out && needs_b(op, 1 - w));
    const uint32_t rm = 1u | (ra ? 2u : 0u) | (rbb ? 4u : 0u);
    RedBuild& rb = S->rb[S->nred];
    const int occ = (op == OP_MUL || op == OP_DIV) ? kOccRedMulDiv : kOccRedAddSub;
    // Cluster plans are built for float storage only.
    const int ock = S->es == 4 ? red_cl_occ(op, true) : 0;
    const int ocr = S->es == 4 ? red_cl_occ(op, false) : 0;
    // div's grad_b carries the factor -1/b^2, applied once to each total.
    const bool post = op == OP_DIV && w == 1;
    rc = build_red(P, xslot, S->g.ptr, ra ? S->a.ptr : nullptr, rbb ? S->b.ptr : nullptr, rm,
                   stream_mask & rm, xo, d_out, 0, occ, ock, ocr, &rb, post);
    if (rc) return rc;
    size_t q = rb.ws_bytes;
    for (int v : {1, 4, 8}) {
      if (v == 8 && S->es != 2) continue;  // 8-wide vectors: bfloat16 only
      RedBuild tmp;
      rc = build_red(P, xslot, S->g.ptr, nullptr, nullptr, rm, 0, xo, d_out, v, occ, ock, ocr,
                     &tmp, post);
      if (rc) return rc;
      q = std::max(q, tmp.ws_bytes);
    }
    S->ws_off[S->nred] = off;
    off += rb.ws_bytes;
    off_q += q;
    S->which[S->nred] = w;
    ++S->nred;
  }
  S->ws_run = off;
  S->ws_query = off_q;
  // Both gradients reduced: one fused pass when the shape allows it.
  if (red_a && red_b && S->es == 4) {
    const int r = build_sab(P, S->g.ptr, S->a.ptr, S->b.ptr, grad_a, grad_b, read_mask, &S->sb,
                            op == OP_DIV);
    if (r == ZR_OK) {
      S->sab = true;
      S->ws_run = S->sb.ws_a_bytes + S->sb.ws_b_bytes;
    } else if (r != 1) {
      return r;
    }
    // The query covers whichever route the run-time pointers select.
    SabBuild any;
    const float* fake = reinterpret_cast<const float*>(uintptr_t(256));
    if (build_sab(P, fake, fake, fake, grad_a, grad_b, read_mask, &any, op == OP_DIV) == ZR_OK)
      S->ws_query = std::max(S->ws_query, any.ws_a_bytes + any.ws_b_bytes);
  }
  return ZR_OK;
}

// ------------------------------------------------------------------ sum to shape

struct SumSet {
  int es = 4;                    // bytes per stored element: 4 float, 2 bfloat16
  bool empty = false;
  bool copy = false;
  EwBuild eb;
  RedBuild rb;
  size_t ws_query = 0;
  float* zero_ptr = nullptr;
  size_t zero_bytes = 0;
  TDesc in, out;
};

int plan_sum(const zr_tensor& tin, int32_t ndo, const int64_t* so, float* out, SumSet* S) {
  int rc = read_tensor(tin, &S->in);
  if (rc) return rc;
  zr_tensor to{out, ndo, so, nullptr};
  if (ndo > 0 && so == nullptr) return ZR_ERR_NULL;
  rc = read_tensor(to, &S->out);
  if (rc) return rc;
  int n = 0;
  int64_t bsz[kMaxDims];
  rc = broadcast_sizes(S->in.nd, S->in.size, S->out.nd, S->out.size, &n, bsz);
  if (rc) return rc;
  if (n != S->in.nd) return ZR_ERR_SHAPE;
  for (int d = 0; d < n; ++d)
    if (bsz[d] != S->in.size[d]) return ZR_ERR_SHAPE;
  const bool reduced = is_reduced(S->out, n, S->in.size);
  const Span sout = span_of(out, S->out.extent, S->es);
  if (overlaps(sout, span_of(S->in.ptr, S->in.extent, S->es)) &&
      (reduced || !same_layout(S->out, S->in)))
    return ZR_ERR_LAYOUT;
  if (S->in.numel == 0) {
    S->empty = true;
    if (S->out.numel > 0) { S->zero_ptr = out; S->zero_bytes = S->out.numel * S->es; }
    return ZR_OK;
  }
  if (!S->in.ptr || !out) return ZR_ERR_NULL;
  int64_t st[kProbSlots][kMaxDims] = {};
  align_strides(S->in, n, S->in.size, st[0]);
  Prob P;
  if (!reduced) {
    S->copy = true;
    int64_t dense[kMaxDims];
    contiguous_strides(n, S->in.size, dense);
    for (int d = 0; d < n; ++d) st[kSlotOut][d] = S->in.size[d] == 1 ? 0 : dense[d];
    rc = coalesce(n, S->in.size, st, 1u | (1u << kSlotOut), -1, &P);
    if (rc) return rc;
    P.es = S->es;
    const float* in[3] = {S->in.ptr, nullptr, nullptr};
    float* outs[2] = {out, nullptr};
    return build_ew(P, in, outs, 1u, 1u, kOccEwCopy, &S->eb);
  }
  grad_index_strides(S->out, n, S->in.size, st[kSlotXA]);
  rc = coalesce(n, S->in.size, st, 1u | (1u << kSlotXA), -1, &P);
  if (rc) return rc;
  P.es = S->es;
  const int ock = S->es == 4 ? red_cl_occ(OP_ADD, true) : 0;
  const int ocr = S->es == 4 ? red_cl_occ(OP_ADD, false) : 0;
  rc = build_red(P, kSlotXA, S->in.ptr, nullptr, nullptr, 1u, 1u, out, nullptr, 0, kOccRedAddSub,
                 ock, ocr, &S->rb);
  if (rc) return rc;
  S->ws_query = S->rb.ws_bytes;
  for (int v : {1, 4, 8}) {
    if (v == 8 && S->es != 2) continue;  // 8-wide vectors: bfloat16 only
    RedBuild tmp;
    rc = build_red(P, kSlotXA, S->in.ptr, nullptr, nullptr, 1u, 0, out, nullptr, v, kOccRedAddSub,
                   ock, ocr, &tmp);
    if (rc) return rc;
    S->ws_query = std::max(S->ws_query, tmp.ws_bytes);
  }
  return ZR_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ZR_OK : ZR_ERR_CUDA; }

// Launch (or, with dry, only guard-check) the kernels of a backward plan.
int launch_bwd_set(const BwdSet& S, int op, void* workspace, cudaStream_t st, bool dry) {
  if (S.direct) return cuda_status(launch_bwd_direct(op, S.want, S.eb, st, dry));
  if (S.sab) {
    SabBuild sb = S.sb;
    sb.plan.ws_a = static_cast<float*>(workspace);
    sb.plan.ws_b = reinterpret_cast<float*>(static_cast<char*>(workspace) + sb.ws_a_bytes);
    return cuda_status(launch_sab(op, sb, st, dry));
  }
  for (int i = 0; i < S.nred; ++i) {
    RedBuild rbi = S.rb[i];
    rbi.plan.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + S.ws_off[i]);
    rbi.comb.partial = rbi.plan.partial;
    const int rc = cuda_status(launch_reduce(op, S.which[i], rbi, st, dry));
    if (rc) return rc;
  }
  return ZR_OK;
}

int launch_sum_set(const SumSet& S, void* workspace, cudaStream_t st, bool dry) {
  if (S.copy) return cuda_status(launch_copy(S.eb, st, dry));
  RedBuild rb = S.rb;
  rb.plan.partial = static_cast<float*>(workspace);
  rb.comb.partial = rb.plan.partial;
  return cuda_status(launch_reduce(OP_ADD, 2, rb, st, dry));
}

int copy_json(const std::string& s, char* buf, size_t len) {
  if (!buf || len == 0) return ZR_ERR_NULL;
  const size_t m = std::min(len - 1, s.size());
  std::memcpy(buf, s.data(), m);
  buf[m] = '\0';
  return ZR_OK;
}


// Plan descriptions (JSON) shared by the test hooks and the trace.
std::string fwd_json(const FwdSet& S) {
  if (S.empty) return "{\"kernel\":\"none\"}";
  if (S.tr) return describe_tr(S.tp);
  if (S.sabf) return describe_sabf(S.sp, S.sp_rpt);
  return describe_ew(S.eb);
}

std::string bwd_json(const BwdSet& S) {
  if (S.nothing || S.empty)
    return "{\"kernel\":\"none\",\"ws_query\":" + std::to_string(S.ws_query) + "}";
  if (S.direct)
    return "{\"plans\":[" + describe_ew(S.eb) + "],\"ws_run\":0,\"ws_query\":" +
           std::to_string(S.ws_query) + "}";
  if (S.sab) {
    const std::string d = describe_sab(S.sb);
    return "{\"plans\":[" + d.substr(0, d.size() - 1) + ",\"nslots\":" +
           std::to_string(S.sb.plan.slots_a) + "}," + d.substr(0, d.size() - 1) + ",\"nslots\":" +
           std::to_string(S.sb.plan.n_tiles) + "}],\"which\":[0,1],\"ws_run\":" +
           std::to_string(S.ws_run) + ",\"ws_query\":" + std::to_string(S.ws_query) + "}";
  }
  std::string s = "{\"plans\":[";
  for (int i = 0; i < S.nred; ++i) {
    if (i) s += ",";
    s += describe_red(S.rb[i]);
  }
  return s + "],\"which\":[" + std::to_string(S.which[0]) +
         (S.nred > 1 ? "," + std::to_string(S.which[1]) : std::string()) +
         "],\"ws_run\":" + std::to_string(S.ws_run) + ",\"ws_query\":" + std::to_string(S.ws_query) +
         "}";
}

std::string sum_json(const SumSet& S) {
  if (S.empty) return "{\"kernel\":\"none\"}";
  if (S.copy) return "{\"plans\":[" + describe_ew(S.eb) + "],\"ws_query\":0}";
  return "{\"plans\":[" + describe_red(S.rb) + "],\"ws_query\":" + std::to_string(S.ws_query) + "}";
}

// ZR_TRACE set (and not "0"): every forward, backward, sum-to-shape and
// unary call that is about to launch writes one line "zr_trace <entry> <plan JSON>" to
// stderr.  Read once per process.
bool trace_on() {
  static const bool on = [] {
    const char* e = std::getenv("ZR_TRACE");
    return e != nullptr && e[0] != '\0' && !(e[0] == '0' && e[1] == '\0');
  }();
  return on;
}

void trace(const char* entry, const std::string& json) {
  std::fprintf(stderr, "zr_trace %s %s\n", entry, json.c_str());
}

}  // namespace
}  // namespace zr

using namespace zr;

extern "C" {

int zr_broadcast_shape(int32_t ndim_a, const int64_t* sizes_a, int32_t ndim_b,
                       const int64_t* sizes_b, int32_t* ndim_out, int64_t sizes_out[ZR_MAX_DIMS]) {
  if (!ndim_out || !sizes_out) return ZR_ERR_NULL;
  if (ndim_a < 0 || ndim_a > kMaxDims || ndim_b < 0 || ndim_b > kMaxDims) return ZR_ERR_RANK;
  if ((ndim_a > 0 && !sizes_a) || (ndim_b > 0 && !sizes_b)) return ZR_ERR_NULL;
  int n = 0;
  int64_t so[kMaxDims];
  const int rc = broadcast_sizes(ndim_a, sizes_a, ndim_b, sizes_b, &n, so);
  if (rc) return rc;
  *ndim_out = n;
  for (int i = 0; i < n; ++i) sizes_out[i] = so[i];
  return ZR_OK;
}

static int binary_fwd_es(int es, zr_op op, zr_tensor a, zr_tensor b, float* out,
                         const int64_t* out_strides, zr_stream_t stream) {
  FwdSet S;
  S.es = es;
  int rc = plan_fwd(op, a, b, out, out_strides, &S);
  if (rc) return rc;
  if (trace_on()) trace("zr_binary_fwd", fwd_json(S));
  if (S.empty) return ZR_OK;
  for (const void* p : {static_cast<const void*>(S.a.ptr), static_cast<const void*>(S.b.ptr),
                        static_cast<const void*>(out)}) {
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  if (S.tr) return cuda_status(launch_fwd_tr(op, S.tp, reinterpret_cast<cudaStream_t>(stream)));
  if (S.sabf)
    return cuda_status(launch_fwd_sabf(op, S.sp_rpt, S.sp, reinterpret_cast<cudaStream_t>(stream)));
  return cuda_status(launch_fwd(op, S.eb, reinterpret_cast<cudaStream_t>(stream)));
}

static int binary_bwd_es(int es, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                         float* grad_a, float* grad_b, void* workspace, size_t* workspace_bytes,
                         zr_stream_t stream) {
  if (!workspace_bytes) return ZR_ERR_NULL;
  BwdSet S;
  S.es = es;
  int rc = plan_bwd(op, grad_out, a, b, grad_a, grad_b, &S);
  if (rc) return rc;
  if (workspace == nullptr) {
    *workspace_bytes = S.ws_query;
    return ZR_OK;
  }
  if (trace_on()) trace("zr_binary_bwd", bwd_json(S));
  if (S.nothing) return ZR_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S.empty) {
    for (int w = 0; w < 2; ++w) {
      if (!S.zero_ptr[w]) continue;
      rc = check_device_ptr(S.zero_ptr[w]);
      if (rc) return rc;
    }
    for (int w = 0; w < 2; ++w)
      if (S.zero_ptr[w] && cudaMemsetAsync(S.zero_ptr[w], 0, S.zero_bytes[w], st) != cudaSuccess)
        return ZR_ERR_CUDA;
    return ZR_OK;
  }
  if (S.ws_run > 0) {
    if (*workspace_bytes < S.ws_run) return ZR_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return ZR_ERR_WORKSPACE;
  }
  // Device checks on every pointer that will be touched.
  const void* ptrs[6] = {S.g.ptr, nullptr, nullptr, grad_a, grad_b,
                         S.ws_run > 0 ? workspace : nullptr};
  const bool ra = (grad_a && needs_a(op, 0)) || (grad_b && needs_a(op, 1));
  const bool rb = (grad_a && needs_b(op, 0)) || (grad_b && needs_b(op, 1));
  if (ra) ptrs[1] = S.a.ptr;
  if (rb) ptrs[2] = S.b.ptr;
  for (const void* p : ptrs) {
    if (!p) continue;
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  return launch_bwd_set(S, op, workspace, st, false);
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation backward
//
// Scratch for zr_binary_bwd_noalloc: the partial sums of its two-pass
// reduction live here instead of in a caller-provided workspace.  The array
// exists once per device that loads this library and stays until the process
// exits.  Host code cannot use the array's name as a device address, so the
// address is looked up with cudaGetSymbolAddress, with the device current, on
// the first call made on it.  The lookup is remembered together with the
// identity of the device's context: a new context (after cudaDeviceReset, for
// example) reloads the module at another address, and the next call then
// looks the address up again instead of launching on a freed one.
static __device__ __align__(256) unsigned char zr_noalloc_scratch[ZR_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kScratchDevices = 256;
struct ScratchAddr {
  void* addr = nullptr;
  unsigned long long ctx = 0;  // context id the address belongs to
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch[kScratchDevices];

// Id of the calling thread's current context (ids are unique for the life of
// the process), through the driver's cuCtxGetId, found at run time so that
// the library does not link the driver library.  False when there is no
// current context or the driver lacks the call.
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
bool current_ctx_id(unsigned long long* id) {
  static const CtxGetIdFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<CtxGetIdFn>(f);
  }();
  return fn != nullptr && fn(nullptr, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ZR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kScratchDevices) return ZR_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& c = g_scratch[dev];
  unsigned long long id = 0;
  const bool have_id = current_ctx_id(&id);
  if (c.addr == nullptr || !have_id || c.ctx != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, zr_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ZR_ERR_CUDA;
    }
    // The lookup makes the device's primary context current if none was.
    // Without a context id the address is not remembered, so every call
    // looks it up.
    c.addr = p;
    c.ctx = 0;
    if (current_ctx_id(&id)) c.ctx = id;
    else c.addr = nullptr;
    *out = p;
    return ZR_OK;
  }
  *out = c.addr;
  return ZR_OK;
}

}  // namespace

extern "C" {

int zr_binary_bwd_noalloc(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b, float* grad_a,
                          float* grad_b, zr_stream_t stream) {
  BwdSet S;
  int rc = plan_bwd(op, grad_out, a, b, grad_a, grad_b, &S);
  if (rc) return rc;
  if (trace_on()) trace("zr_binary_bwd_noalloc", bwd_json(S));
  if (S.nothing) return ZR_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S.empty) {
    for (int w = 0; w < 2; ++w) {
      if (!S.zero_ptr[w]) continue;
      rc = check_device_ptr(S.zero_ptr[w]);
      if (rc) return rc;
    }
    for (int w = 0; w < 2; ++w)
      if (S.zero_ptr[w] && cudaMemsetAsync(S.zero_ptr[w], 0, S.zero_bytes[w], st) != cudaSuccess)
        return ZR_ERR_CUDA;
    return ZR_OK;
  }
  // The plan's partials must fit the fixed scratch array.
  if (S.ws_run > size_t(ZR_STATIC_SCRATCH_BYTES)) return ZR_ERR_WORKSPACE;
  const bool ra = (grad_a && needs_a(op, 0)) || (grad_b && needs_a(op, 1));
  const bool rb = (grad_a && needs_b(op, 0)) || (grad_b && needs_b(op, 1));
  const void* ptrs[5] = {S.g.ptr, ra ? S.a.ptr : nullptr, rb ? S.b.ptr : nullptr, grad_a, grad_b};
  for (const void* p : ptrs) {
    if (!p) continue;
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  void* scratch = nullptr;
  if (S.ws_run > 0) {
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
  }
  // Every partial slot the plan uses is written by the first pass before the
  // second pass reads it, so the scratch needs no clearing between calls.
  return launch_bwd_set(S, op, scratch, st, false);
}

static int sum_to_shape_es(int es, zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                           float* out, void* workspace, size_t* workspace_bytes,
                           zr_stream_t stream) {
  if (!workspace_bytes) return ZR_ERR_NULL;
  SumSet S;
  S.es = es;
  int rc = plan_sum(in, ndim_out, sizes_out, out, &S);
  if (rc) return rc;
  if (workspace == nullptr) {
    *workspace_bytes = S.ws_query;
    return ZR_OK;
  }
  if (trace_on()) trace("zr_sum_to_shape", sum_json(S));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S.empty) {
    if (!S.zero_ptr) return ZR_OK;
    rc = check_device_ptr(S.zero_ptr);
    if (rc) return rc;
    return cuda_status(cudaMemsetAsync(S.zero_ptr, 0, S.zero_bytes, st));
  }
  const size_t need = S.copy ? 0 : S.rb.ws_bytes;
  if (need > 0) {
    if (*workspace_bytes < need) return ZR_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return ZR_ERR_WORKSPACE;
  }
  for (const void* p : {static_cast<const void*>(S.in.ptr), static_cast<const void*>(out),
                        need > 0 ? static_cast<const void*>(workspace) : nullptr}) {
    if (!p) continue;
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  return launch_sum_set(S, workspace, st, false);
}

int zr_binary_fwd(zr_op op, zr_tensor a, zr_tensor b, float* out, const int64_t* out_strides,
                  zr_stream_t stream) {
  return binary_fwd_es(4, op, a, b, out, out_strides, stream);
}

int zr_binary_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b, float* grad_a,
                  float* grad_b, void* workspace, size_t* workspace_bytes, zr_stream_t stream) {
  return binary_bwd_es(4, op, grad_out, a, b, grad_a, grad_b, workspace, workspace_bytes, stream);
}

int zr_sum_to_shape(zr_tensor in, int32_t ndim_out, const int64_t* sizes_out, float* out,
                    void* workspace, size_t* workspace_bytes, zr_stream_t stream) {
  return sum_to_shape_es(4, in, ndim_out, sizes_out, out, workspace, workspace_bytes, stream);
}

static int dtype_bytes(int dtype) { return dtype == ZR_F32 ? 4 : (dtype == ZR_BF16 ? 2 : 0); }

int zr_binary_fwd_t(zr_dtype dtype, zr_op op, zr_tensor a, zr_tensor b, void* out,
                    const int64_t* out_strides, zr_stream_t stream) {
  const int es = dtype_bytes(dtype);
  if (!es) return ZR_ERR_DTYPE;
  return binary_fwd_es(es, op, a, b, static_cast<float*>(out), out_strides, stream);
}

int zr_binary_bwd_t(zr_dtype dtype, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                    void* grad_a, void* grad_b, void* workspace, size_t* workspace_bytes,
                    zr_stream_t stream) {
  const int es = dtype_bytes(dtype);
  if (!es) return ZR_ERR_DTYPE;
  return binary_bwd_es(es, op, grad_out, a, b, static_cast<float*>(grad_a),
                       static_cast<float*>(grad_b), workspace, workspace_bytes, stream);
}

int zr_sum_to_shape_t(zr_dtype dtype, zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                      void* out, void* workspace, size_t* workspace_bytes, zr_stream_t stream) {
  const int es = dtype_bytes(dtype);
  if (!es) return ZR_ERR_DTYPE;
  return sum_to_shape_es(es, in, ndim_out, sizes_out, static_cast<float*>(out), workspace,
                         workspace_bytes, stream);
}

const char* zr_status_string(int status) {
  switch (status) {
    case ZR_OK: return "ZR_OK";
    case ZR_ERR_DTYPE: return "ZR_ERR_DTYPE: unknown element type";
    case ZR_ERR_NULL: return "ZR_ERR_NULL: required pointer is NULL or op code unknown";
    case ZR_ERR_RANK: return "ZR_ERR_RANK: ndim < 0 or ndim > 8";
    case ZR_ERR_SHAPE: return "ZR_ERR_SHAPE: shapes not broadcastable or wrong grad_out shape";
    case ZR_ERR_SIZE: return "ZR_ERR_SIZE: negative size or stride, or index range overflow";
    case ZR_ERR_LAYOUT: return "ZR_ERR_LAYOUT: output overlaps itself, an input or another output";
    case ZR_ERR_DEVICE: return "ZR_ERR_DEVICE: pointer not addressable by the current device";
    case ZR_ERR_WORKSPACE: return "ZR_ERR_WORKSPACE: workspace too small or misaligned";
    case ZR_ERR_CUDA: return "ZR_ERR_CUDA: CUDA call or kernel launch failed";
    default: return "unknown zr status";
  }
}

// ------------------------------------------------------------------ test hooks

int zr_test_fastdiv(uint32_t d, uint32_t n, uint32_t* q) {
  if (!q || d == 0) return ZR_ERR_NULL;
  *q = fd_div(make_fastdiv(d), n);
  return ZR_OK;
}

int zr_test_dry_run_fwd(zr_op op, zr_tensor a, zr_tensor b, const float* out,
                        const int64_t* out_strides) {
  FwdSet S;
  const int rc = plan_fwd(op, a, b, out, out_strides, &S);
  if (rc || S.empty) return rc;
  if (S.tr) return cuda_status(launch_fwd_tr(op, S.tp, nullptr, true));
  if (S.sabf) return cuda_status(launch_fwd_sabf(op, S.sp_rpt, S.sp, nullptr, true));
  return cuda_status(launch_fwd(op, S.eb, nullptr, true));
}

int zr_test_dry_run_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                        const float* grad_a, const float* grad_b) {
  BwdSet S;
  const int rc = plan_bwd(op, grad_out, a, b, const_cast<float*>(grad_a),
                          const_cast<float*>(grad_b), &S);
  if (rc || S.nothing || S.empty) return rc;
  // A stand-in workspace address: only checked for presence, never touched.
  return launch_bwd_set(S, op, reinterpret_cast<void*>(uintptr_t(1) << 40), nullptr, true);
}

int zr_test_occupancy(int which, int* planned, int* actual) {
  if (!planned || !actual) return ZR_ERR_NULL;
  cudaError_t e;
  if (which >= 0 && which < 4) e = occupancy_ew(which, planned, actual);
  else if (which >= 4 && which < 9) e = occupancy_red(which - 4, planned, actual);
  else if (which >= 9 && which < 11) e = occupancy_other(which - 9, planned, actual);
  else if (which >= 11 && which < 16) e = occupancy_red(which - 6, planned, actual);
  else if (which >= 16 && which < 20) e = occupancy_chain(which - 16, planned, actual);
  else if (which >= 20 && which < 22) e = occupancy_ew(which - 16, planned, actual);
  else if (which >= 22 && which < 24) e = occupancy_ew(which - 16, planned, actual);
  else if (which == 24) e = occupancy_bf16(0, planned, actual);
  else if (which == 25) e = occupancy_red(10, planned, actual);
  else if (which >= 26 && which < 28) e = occupancy_bf16(which - 25, planned, actual);
  else return ZR_ERR_SIZE;
  return cuda_status(e);
}

int zr_test_div_short_check(unsigned long long* out, void* stream) {
  const int rc = check_device_ptr(out);
  if (rc) return rc;
  return cuda_status(launch_div_short_check(out, static_cast<cudaStream_t>(stream)));
}

int zr_test_dry_run_sum(zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                        const float* out) {
  SumSet S;
  const int rc = plan_sum(in, ndim_out, sizes_out, const_cast<float*>(out), &S);
  if (rc || S.empty) return rc;
  return launch_sum_set(S, reinterpret_cast<void*>(uintptr_t(1) << 40), nullptr, true);
}

int zr_test_describe_fwd(zr_op op, zr_tensor a, zr_tensor b, const float* out,
                         const int64_t* out_strides, char* buf, size_t len) {
  FwdSet S;
  const int rc = plan_fwd(op, a, b, out, out_strides, &S);
  if (rc) return rc;
  return copy_json(fwd_json(S), buf, len);
}

int zr_test_describe_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                         const float* grad_a, const float* grad_b, char* buf, size_t len) {
  return zr_test_describe_bwd_t(ZR_F32, op, grad_out, a, b, grad_a, grad_b, buf, len);
}

int zr_test_describe_bwd_t(zr_dtype dtype, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                           const void* grad_a, const void* grad_b, char* buf, size_t len) {
  if (dtype != ZR_F32 && dtype != ZR_BF16) return ZR_ERR_DTYPE;
  BwdSet S;
  S.es = dtype == ZR_BF16 ? 2 : 4;
  const int rc = plan_bwd(op, grad_out, a, b, static_cast<float*>(const_cast<void*>(grad_a)),
                          static_cast<float*>(const_cast<void*>(grad_b)), &S);
  if (rc) return rc;
  return copy_json(bwd_json(S), buf, len);
}

int zr_test_describe_sum(zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                         const float* out, char* buf, size_t len) {
  SumSet S;
  const int rc = plan_sum(in, ndim_out, sizes_out, const_cast<float*>(out), &S);
  if (rc) return rc;
  return copy_json(sum_json(S), buf, len);
}

}  // extern "C"

namespace zr {
namespace {

// Host walk of k_elementwise's (CTA, item, lane) space, or k_flat's for a
// flat plan.
template <class Rec>
void walk_ew(const EwBuild& eb, Rec rec) {
  const EwPlan& p = eb.plan;
  if (p.flat) {
    for (uint32_t cta = 0; cta < p.n_cta; ++cta) {
      const uint32_t first = cta * p.items_per_cta;
      const uint32_t left = p.nitems - first;
      const uint32_t end = first + (left < p.items_per_cta ? left : p.items_per_cta);
      for (uint32_t it0 = first; it0 < end; it0 += 4 * kThreads)
        for (uint32_t u = 0; u < 4; ++u)
          for (uint32_t t = 0; t < uint32_t(kThreads); ++t) {
            const uint32_t item = it0 + u * kThreads + t;
            if (item >= end) continue;
            const uint32_t row = fd_div(p.nvcol_div, item);
            const uint32_t vc = item - row * p.nvcol;
            for (int i = 0; i < eb.vec; ++i) {
              const int64_t c = int64_t(vc) * eb.vec + i;
              if (c >= p.ncol) continue;
              int64_t o[kMaxOperands];
              for (int k = 0; k < kMaxOperands; ++k)
                o[k] = int64_t(row) * p.rows.stride[k][0] + c * p.inner_stride[k];
              rec(o);
            }
          }
    }
    return;
  }
  for (uint32_t cta = 0; cta < p.n_cta; ++cta) {
    const EwTile t = ew_tile(p, cta);
    for (uint32_t item = 0; item < p.items_per_cta; ++item) {
      const uint32_t ri = fd_div(p.tile_vcols_div, item);
      const uint32_t vc = item - ri * p.tile_vcols;
      if (!(ri < t.nrows && vc < t.nvcols)) continue;
      int64_t off[kMaxOperands];
      decomp_offsets(p.rows, t.row0 + ri, off);
      for (int i = 0; i < eb.vec; ++i) {
        const int64_t c = int64_t(t.vcol0 + vc) * eb.vec + i;
        if (c >= p.ncol) continue;
        int64_t o[kMaxOperands];
        for (int k = 0; k < kMaxOperands; ++k) o[k] = off[k] + c * p.inner_stride[k];
        rec(o);
      }
    }
  }
}

// Host walk of k_transpose's (CTA, p, q) space; o[0] = x, o[1] = y, o[3] = out.
template <class Rec>
void walk_tr(const TrPlan& p, Rec rec) {
  for (uint32_t cta = 0; cta < p.n_cta; ++cta) {
    const uint32_t t1 = fd_div(p.n_qt_div, cta);
    const uint32_t qt = cta - t1 * p.n_qt;
    const uint32_t bidx = fd_div(p.n_pt_div, t1);
    const uint32_t pt = t1 - bidx * p.n_pt;
    int64_t base[kMaxOperands];
    decomp_offsets(p.batch, bidx, base);
    // Thread (warp w, lane) covers p = 16w + 4(lane & 3) + c, q = 4(lane >> 2) + k.
    for (uint32_t t = 0; t < kThreads; ++t) {
      const uint32_t w = t >> 5, lane = t & 31;
      for (uint32_t c = 0; c < 4; ++c)
      for (uint32_t k = 0; k < 4; ++k) {
        const uint32_t pp = pt * kTrP + 16 * w + 4 * (lane & 3) + c;
        const uint32_t q = qt * kTrTile + 4 * (lane >> 2) + k;
        if (q >= p.nq || pp >= p.np) continue;
        int64_t o[kMaxOperands] = {base[0] + pp + int64_t(q) * p.xs_q,
                                   base[1] + int64_t(pp) * p.ys_p + int64_t(q) * p.ys_q, 0,
                                   base[kSlotOut] + int64_t(pp) * p.os_p + q};
        rec(o);
      }
    }
  }
}

// Host walk of k_sabf's (CTA, row, beta, column) space; o[0] = a, o[1] = b,
// o[3] = out.
template <class Rec>
void walk_sabf(const SabFPlan& p, Rec rec) {
  for (uint32_t cta = 0; cta < p.n_cta; ++cta) {
    const uint32_t tile = fd_div(p.n_bc_div, cta);
    const uint32_t bc = cta - tile * p.n_bc;
    int64_t ob[kMaxOperands];
    decomp_offsets(p.a_outer, tile, ob);
    const uint32_t b0 = bc * p.beta_chunk, b1 = std::min(p.n_beta, b0 + p.beta_chunk);
    for (uint32_t r = 0; r < p.ta; ++r) {
      int64_t ri[kMaxOperands];
      decomp_offsets(p.a_inner, r, ri);
      for (uint32_t beta = b0; beta < b1; ++beta) {
        int64_t bo[kMaxOperands];
        decomp_offsets(p.beta, beta, bo);
        for (uint32_t c = 0; c < p.ncol; ++c) {
          int64_t o[kMaxOperands] = {ob[1] + ri[1] + c, bo[2] + c, 0, ob[0] + ri[0] + bo[0] + c};
          rec(o);
        }
      }
    }
  }
}

// Host walk of k_reduce's (CTA, row, column, lane) space.
template <class Rec>
void walk_red(const RedBuild& rb, Rec rec) {
  const RedPlan& p = rb.plan;
  for (uint32_t cta = 0; cta < p.n_cta; ++cta) {
    const RedCta c = red_cta(p, cta);
    int64_t base[kMaxOperands];
    decomp_offsets(p.kept, c.kidx, base);
    const uint32_t row0 = c.rblk * p.rows_per_blk;
    const uint32_t nrows = std::min(p.rows_per_blk, p.n_red - row0);
    const uint32_t vb = c.cblk * p.vcols_per_blk;
    const uint32_t ve = std::min(vb + p.vcols_per_blk, p.nvcol);
    for (uint32_t r = 0; r < nrows; ++r) {
      int64_t off[kMaxOperands];
      decomp_offsets(p.red, row0 + r, off);
      for (uint32_t vc = vb; vc < ve; ++vc) {
        for (int i = 0; i < rb.vec; ++i) {
          const int64_t col = int64_t(vc) * rb.vec + i;
          if (col >= p.ncol) continue;
          int64_t o[kMaxOperands];
          for (int k = 0; k < kMaxOperands; ++k) o[k] = base[k] + off[k] + col * p.inner_stride[k];
          const int64_t x = p.inner_kept ? int64_t(c.kidx) * p.ncol + col : int64_t(c.kidx);
          const int64_t slot = p.inner_kept ? c.rblk : int64_t(c.rblk) * p.n_cblk + c.cblk;
          rec(o, x, slot);
        }
      }
    }
  }
}

// Host walk of k_sab's (CTA, step, row, column) space.  rec(o, x_a, slot_a,
// x_b, slot_b).  Also replays the grad_a flushes and zero fills and returns
// false unless every (slot, tile) pair is written exactly once.
template <class Rec>
bool walk_sab(const SabBuild& sb, Rec rec) {
  const SabPlan& p = sb.plan;
  std::vector<int> writes(size_t(p.n_tiles) * p.slots_a, 0);
  std::vector<int64_t> row_g(p.ta), row_a(p.ta), beta_g(p.n_beta), beta_b(p.n_beta);
  for (uint32_t i = 0; i < p.ta; ++i) {
    int64_t off[kMaxOperands];
    decomp_offsets(p.a_inner, i, off);
    row_g[i] = off[0];
    row_a[i] = off[1];
  }
  for (uint32_t i = 0; i < p.n_beta; ++i) {
    int64_t off[kMaxOperands];
    decomp_offsets(p.beta, i, off);
    beta_g[i] = off[0];
    beta_b[i] = off[2];
  }
  for (uint32_t c = 0; c < p.grid; ++c) {
    const uint64_t s0 = sab_start(p, c), s1 = sab_start(p, c + 1);
    for (uint64_t step = s0; step < s1; ++step) {
      const uint32_t tile = fd_div(p.n_beta_div, uint32_t(step));
      const uint32_t beta = uint32_t(step) - tile * p.n_beta;
      int64_t ob[kMaxOperands];
      decomp_offsets(p.a_outer, tile, ob);
      const uint32_t slot = c - sab_owner(p, uint64_t(tile) * p.n_beta);
      for (uint32_t r = 0; r < p.ta; ++r) {
        for (uint32_t col = 0; col < p.ncol; ++col) {
          int64_t o[kMaxOperands] = {ob[0] + row_g[r] + beta_g[beta] + col,
                                     ob[1] + row_a[r] + col, beta_b[beta] + col, -1};
          rec(o, (int64_t(tile) * p.ta + r) * p.ncol + col, int64_t(slot),
              int64_t(beta) * p.ncol + col, int64_t(tile));
        }
      }
      if (beta == p.n_beta - 1 || step == s1 - 1) {
        if (slot >= p.slots_a) return false;
        writes[size_t(tile) * p.slots_a + slot]++;
        if (beta == p.n_beta - 1)
          for (uint32_t s = slot + 1; s < p.slots_a; ++s) writes[size_t(tile) * p.slots_a + s]++;
      }
    }
  }
  for (int w : writes)
    if (w != 1) return false;
  return true;
}

}  // namespace
}  // namespace zr

extern "C" {

int zr_test_emulate_fwd(zr_tensor a, zr_tensor b, const float* out, const int64_t* out_strides,
                        int64_t cap, int64_t* rec, int64_t* nrec) {
  return zr_test_emulate_fwd_t(ZR_F32, a, b, out, out_strides, cap, rec, nrec);
}

int zr_test_emulate_fwd_t(zr_dtype dtype, zr_tensor a, zr_tensor b, const void* out,
                          const int64_t* out_strides, int64_t cap, int64_t* rec, int64_t* nrec) {
  if (!rec || !nrec) return ZR_ERR_NULL;
  if (dtype != ZR_F32 && dtype != ZR_BF16) return ZR_ERR_DTYPE;
  FwdSet S;
  S.es = dtype == ZR_BF16 ? 2 : 4;
  const int rc = plan_fwd(OP_ADD, a, b, static_cast<const float*>(out), out_strides, &S);
  if (rc) return rc;
  int64_t m = 0;
  bool over = false;
  if (!S.empty && S.tr) {
    walk_tr(S.tp, [&](const int64_t* o) {
      if (m >= cap) { over = true; return; }
      rec[3 * m + 0] = o[kSlotOut];
      rec[3 * m + 1] = S.tp.x_is_a ? o[0] : o[1];
      rec[3 * m + 2] = S.tp.x_is_a ? o[1] : o[0];
      ++m;
    });
  } else if (!S.empty && S.sabf) {
    walk_sabf(S.sp, [&](const int64_t* o) {
      if (m >= cap) { over = true; return; }
      rec[3 * m + 0] = o[kSlotOut];
      rec[3 * m + 1] = o[0];
      rec[3 * m + 2] = o[1];
      ++m;
    });
  } else if (!S.empty) {
    walk_ew(S.eb, [&](const int64_t* o) {
      if (m >= cap) { over = true; return; }
      rec[3 * m + 0] = o[kSlotOut];
      rec[3 * m + 1] = o[0];
      rec[3 * m + 2] = o[1];
      ++m;
    });
  }
  *nrec = m;
  return over ? ZR_ERR_SIZE : ZR_OK;
}

int zr_test_emulate_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                        const float* grad_a, const float* grad_b, int64_t cap, int64_t* rec,
                        int64_t* nrec) {
  return zr_test_emulate_bwd_t(ZR_F32, op, grad_out, a, b, grad_a, grad_b, cap, rec, nrec);
}

int zr_test_emulate_bwd_t(zr_dtype dtype, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                          const void* grad_a, const void* grad_b, int64_t cap, int64_t* rec,
                          int64_t* nrec) {
  if (!rec || !nrec) return ZR_ERR_NULL;
  if (dtype != ZR_F32 && dtype != ZR_BF16) return ZR_ERR_DTYPE;
  BwdSet S;
  S.es = dtype == ZR_BF16 ? 2 : 4;
  const int rc = plan_bwd(op, grad_out, a, b, static_cast<float*>(const_cast<void*>(grad_a)),
                          static_cast<float*>(const_cast<void*>(grad_b)), &S);
  if (rc) return rc;
  int64_t m = 0;
  bool over = false;
  auto put = [&](int64_t plan, const int64_t* o, uint32_t rmask, int64_t x, int64_t slot,
                 bool has_d) {
    if (m >= cap) { over = true; return; }
    int64_t* r = rec + 7 * m;
    r[0] = plan;
    r[1] = o[0];
    r[2] = (rmask & 2) ? o[1] : -1;
    r[3] = (rmask & 4) ? o[2] : -1;
    r[4] = x;
    r[5] = slot;
    r[6] = has_d ? o[kSlotOut] : -1;
    ++m;
  };
  if (!S.nothing && !S.empty) {
    if (S.sab) {
      const uint32_t rm = 1u | (S.sb.plan.a ? 2u : 0u) | (S.sb.plan.b ? 4u : 0u);
      const bool ok = walk_sab(S.sb, [&](const int64_t* o, int64_t xa, int64_t sa, int64_t xb,
                                         int64_t sbs) {
        put(0, o, rm, xa, sa, false);
        put(1, o, rm, xb, sbs, false);
      });
      if (!ok) return ZR_ERR_CUDA;
    } else if (S.direct) {
      const uint32_t rm = 1u | (S.eb.plan.in[1] && ((S.want & 2) && needs_a(op, 1)) ? 2u : 0u) |
                          (S.eb.plan.in[2] && (((S.want & 1) && needs_b(op, 0)) ||
                                               ((S.want & 2) && needs_b(op, 1))) ? 4u : 0u);
      walk_ew(S.eb, [&](const int64_t* o) { put(0, o, rm, -1, -1, true); });
    } else {
      for (int i = 0; i < S.nred; ++i) {
        const RedPlan& p = S.rb[i].plan;
        const uint32_t rm = 1u | (p.a ? 2u : 0u) | (p.b ? 4u : 0u);
        walk_red(S.rb[i], [&](const int64_t* o, int64_t x, int64_t slot) {
          put(i, o, rm, x, slot, p.d_out != nullptr);
        });
      }
    }
  }
  *nrec = m;
  return over ? ZR_ERR_SIZE : ZR_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ two-op chains
//
// out = (a op1 b) op2 c (Operator page, section 融合: one launch and no
// round trip of the intermediate through memory; the mathematics is that of
// the two operators in sequence).  The forward is one elementwise pass.  The
// backward runs as one fused pass when a has the output's shape, b is
// reduced and c either has b's dense layout or one element; any other layout
// runs the composition: t = a op1 b and grad_t in the workspace, then op2's
// and op1's backward passes.

namespace zr {
namespace {

struct ChainFwdSet {
  bool empty = false;
  bool c_one = false;  // c has one element
  EwBuild eb;
  TDesc a, b, c, out;
};

int plan_chain_fwd(int op1, int op2, const zr_tensor& ta, const zr_tensor& tb,
                   const zr_tensor& tc, const float* out, const int64_t* out_strides,
                   ChainFwdSet* S) {
  if (!op_ok(op1) || !op_ok(op2)) return ZR_ERR_NULL;
  int rc = read_tensor(ta, &S->a);
  if (rc) return rc;
  rc = read_tensor(tb, &S->b);
  if (rc) return rc;
  rc = read_tensor(tc, &S->c);
  if (rc) return rc;
  int nt = 0, n = 0;
  int64_t szt[kMaxDims], osz[kMaxDims];
  rc = broadcast_sizes(S->a.nd, S->a.size, S->b.nd, S->b.size, &nt, szt);
  if (rc) return rc;
  rc = broadcast_sizes(nt, szt, S->c.nd, S->c.size, &n, osz);
  if (rc) return rc;
  zr_tensor to{out, n, osz, out_strides};
  rc = read_tensor(to, &S->out);
  if (rc) return rc;
  if (S->out.numel == 0) {
    S->empty = true;
    return ZR_OK;
  }
  if (!S->a.ptr || !S->b.ptr || !S->c.ptr || !out) return ZR_ERR_NULL;
  if (!non_overlapping(S->out)) return ZR_ERR_LAYOUT;
  const Span so = span_of(out, S->out.extent);
  for (const TDesc* x : {&S->a, &S->b, &S->c})
    if (overlaps(so, span_of(x->ptr, x->extent)) && !same_layout(*x, S->out)) return ZR_ERR_LAYOUT;
  int64_t st[kProbSlots][kMaxDims] = {};
  align_strides(S->a, n, osz, st[0]);
  align_strides(S->b, n, osz, st[1]);
  align_strides(S->c, n, osz, st[2]);
  for (int d = 0; d < n; ++d) st[kSlotOut][d] = osz[d] == 1 ? 0 : S->out.stride[d];
  Prob P;
  rc = coalesce(n, osz, st, 0x7u | (1u << kSlotOut), kSlotOut, &P);
  if (rc) return rc;
  const float* in[3] = {S->a.ptr, S->b.ptr, S->c.ptr};
  float* outs[2] = {const_cast<float*>(out), nullptr};
  const uint32_t stream_mask = (S->a.numel == S->out.numel ? 1u : 0u) |
                               (S->b.numel == S->out.numel ? 2u : 0u) |
                               (S->c.numel == S->out.numel ? 4u : 0u);
  S->c_one = S->c.numel == 1;
  return build_ew(P, in, outs, 0x7u, stream_mask, S->c_one ? kOccEwFwd : kOccEwBwd, &S->eb);
}

struct ChainBwdSet {
  bool nothing = false;
  bool empty = false;
  float* zero_ptr[3] = {nullptr, nullptr, nullptr};
  size_t zero_bytes[3] = {0, 0, 0};
  bool fused = false;
  ChainBuild cb;
  size_t off_c = 0;             // fused: grad_c partial region
  // Composed route: t (when op2's grad_c needs it) and grad_t in the
  // workspace, then op2's and op1's backward passes sharing one partial
  // region (they run in stream order).
  bool need_t = false, need_gt = false;
  FwdSet tf;
  BwdSet b2, b1;
  size_t off_gt = 0, off_p = 0;
  size_t ws_run = 0, ws_query = 0;
  TDesc g, a, b, c;
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

bool dense_layout(const TDesc& t) {
  int64_t want = 1;
  for (int d = t.nd - 1; d >= 0; --d) {
    if (t.size[d] != 1 && t.stride[d] != want) return false;
    want *= t.size[d];
  }
  return true;
}

// Sizes of x right-aligned to rank n (missing dims are 1).
void aligned_sizes(const TDesc& x, int n, int64_t* out) {
  for (int d = 0; d < n; ++d) {
    const int k = d - (n - x.nd);
    out[d] = k < 0 ? 1 : x.size[k];
  }
}

// Plans of the composed route with the workspace at `base` (a real
// workspace, or at query time an address range above every operand so that
// the layout checks see no overlap).
int plan_chain_composed(int op1, int op2, const zr_tensor& tg, const zr_tensor& ta,
                        const zr_tensor& tb, const zr_tensor& tc, float* grad_a, float* grad_b,
                        float* grad_c, int nt, const int64_t* szt, int64_t numel_t, char* base,
                        ChainBwdSet* S, size_t* ws_run, size_t* ws_query) {
  const size_t t_bytes = S->need_t ? align256(size_t(numel_t) * 4) : 0;
  const size_t gt_bytes = S->need_gt ? align256(size_t(numel_t) * 4) : 0;
  S->off_gt = t_bytes;
  S->off_p = t_bytes + gt_bytes;
  float* tptr = reinterpret_cast<float*>(base);
  float* gtptr = reinterpret_cast<float*>(base + S->off_gt);
  int rc;
  if (S->need_t) {
    rc = plan_fwd(op1, ta, tb, tptr, nullptr, &S->tf);
    if (rc) return rc;
  }
  const zr_tensor tt{S->need_t ? tptr : nullptr, nt, szt, nullptr};
  rc = plan_bwd(op2, tg, tt, tc, S->need_gt ? gtptr : nullptr, grad_c, &S->b2);
  if (rc) return rc;
  size_t run = S->b2.ws_run, query = S->b2.ws_query;
  if (S->need_gt) {
    const zr_tensor tgt{gtptr, nt, szt, nullptr};
    rc = plan_bwd(op1, tgt, ta, tb, grad_a, grad_b, &S->b1);
    if (rc) return rc;
    run = std::max(run, S->b1.ws_run);
    query = std::max(query, S->b1.ws_query);
  }
  *ws_run = S->off_p + run;
  *ws_query = S->off_p + query;
  return ZR_OK;
}

int plan_chain_bwd(int op1, int op2, const zr_tensor& tg, const zr_tensor& ta, const zr_tensor& tb,
                   const zr_tensor& tc, float* grad_a, float* grad_b, float* grad_c,
                   void* workspace, ChainBwdSet* S) {
  if (!op_ok(op1) || !op_ok(op2)) return ZR_ERR_NULL;
  int rc = read_tensor(tg, &S->g);
  if (rc) return rc;
  rc = read_tensor(ta, &S->a);
  if (rc) return rc;
  rc = read_tensor(tb, &S->b);
  if (rc) return rc;
  rc = read_tensor(tc, &S->c);
  if (rc) return rc;
  int nt = 0, n = 0;
  int64_t szt[kMaxDims], osz[kMaxDims];
  rc = broadcast_sizes(S->a.nd, S->a.size, S->b.nd, S->b.size, &nt, szt);
  if (rc) return rc;
  rc = broadcast_sizes(nt, szt, S->c.nd, S->c.size, &n, osz);
  if (rc) return rc;
  if (S->g.nd != n) return ZR_ERR_SHAPE;
  for (int d = 0; d < n; ++d)
    if (S->g.size[d] != osz[d]) return ZR_ERR_SHAPE;
  if (!grad_a && !grad_b && !grad_c) {
    S->nothing = true;
    return ZR_OK;
  }
  int64_t numel_t = 1;
  for (int d = 0; d < nt; ++d) numel_t *= szt[d];
  // Layout: the gradients are dense in their inputs' shapes, disjoint from
  // one another and from every input.
  const TDesc ga = dense_desc(grad_a, S->a.nd, S->a.size);
  const TDesc gb = dense_desc(grad_b, S->b.nd, S->b.size);
  const TDesc gc = dense_desc(grad_c, S->c.nd, S->c.size);
  const Span sg[3] = {span_of(grad_a, ga.extent), span_of(grad_b, gb.extent),
                      span_of(grad_c, gc.extent)};
  for (int i = 0; i < 3; ++i) {
    for (int k = i + 1; k < 3; ++k)
      if (overlaps(sg[i], sg[k])) return ZR_ERR_LAYOUT;
    for (const TDesc* x : {&S->g, &S->a, &S->b, &S->c})
      if (overlaps(sg[i], span_of(x->ptr, x->extent))) return ZR_ERR_LAYOUT;
  }
  if (S->g.numel == 0) {
    S->empty = true;
    float* gp[3] = {grad_a, grad_b, grad_c};
    const TDesc* gd[3] = {&ga, &gb, &gc};
    for (int i = 0; i < 3; ++i)
      if (gp[i] && gd[i]->numel > 0) { S->zero_ptr[i] = gp[i]; S->zero_bytes[i] = gd[i]->numel * 4; }
    return ZR_OK;
  }
  // Operands the requested gradients read.
  S->need_t = grad_c && (op2 == OP_MUL || op2 == OP_DIV);
  S->need_gt = grad_a || grad_b;
  const bool read_a = S->need_t || (grad_b && needs_a(op1, 1));
  const bool read_b = S->need_t || (grad_a && needs_b(op1, 0)) || (grad_b && needs_b(op1, 1));
  const bool read_c = (S->need_gt && needs_b(op2, 0)) || (grad_c && needs_b(op2, 1));
  if (!S->g.ptr || (read_a && !S->a.ptr) || (read_b && !S->b.ptr) || (read_c && !S->c.ptr))
    return ZR_ERR_NULL;

  // Fused route: a has the output's shape, b is reduced, and c has b's dense
  // layout or one element; every gradient requested and every operand given.
  size_t fused_q = 0;
  bool shape_ok = grad_a && grad_b && grad_c && S->a.ptr && S->b.ptr && S->c.ptr &&
                  S->a.numel == S->g.numel && S->b.numel < S->g.numel;
  bool c_scalar = S->c.numel == 1;
  if (shape_ok && !c_scalar) {
    int64_t sb[kMaxDims], sc[kMaxDims];
    aligned_sizes(S->b, n, sb);
    aligned_sizes(S->c, n, sc);
    for (int d = 0; d < n; ++d) shape_ok = shape_ok && sb[d] == sc[d];
    shape_ok = shape_ok && dense_layout(S->b) && dense_layout(S->c);
  }
  if (shape_ok) {
    int64_t st[kProbSlots][kMaxDims] = {};
    align_strides(S->g, n, osz, st[0]);
    align_strides(S->a, n, osz, st[1]);
    align_strides(S->b, n, osz, st[2]);
    int64_t dense[kMaxDims];
    contiguous_strides(n, osz, dense);
    for (int d = 0; d < n; ++d) st[kSlotOut][d] = osz[d] == 1 ? 0 : dense[d];
    grad_index_strides(S->b, n, osz, st[kSlotXB]);
    Prob P;
    rc = coalesce(n, osz, st, 0x7u | (1u << kSlotOut) | (1u << kSlotXB), -1, &P);
    if (rc) return rc;
    const uint32_t stream_mask = 1u | 2u | (S->b.numel == S->g.numel ? 4u : 0u);
    ChainBuild q;
    const bool div1 = op1 == OP_DIV, div2 = op2 == OP_DIV;
    if (build_chain(P, S->g.ptr, S->a.ptr, S->b.ptr, S->c.ptr, c_scalar, grad_a, grad_b, grad_c,
                    stream_mask, 4, &q, div1, div2) == ZR_OK)
      fused_q = align256(q.ws_b_bytes) + q.ws_c_bytes;
    const int r = build_chain(P, S->g.ptr, S->a.ptr, S->b.ptr, S->c.ptr, c_scalar, grad_a,
                              grad_b, grad_c, stream_mask, 0, &S->cb, div1, div2);
    if (r == ZR_OK) {
      S->fused = true;
      S->off_c = align256(S->cb.ws_b_bytes);
      S->ws_run = S->off_c + S->cb.ws_c_bytes;
    } else if (r != 1) {
      return r;
    }
  }

  // Composed route: sized for the query always, planned on the real
  // workspace when it runs.
  uintptr_t top = 0;
  for (const TDesc* x : {&S->g, &S->a, &S->b, &S->c}) {
    const Span sp = span_of(x->ptr, x->extent);
    top = std::max(top, sp.hi);
  }
  for (const Span& sp : sg) top = std::max(top, sp.hi);
  char* fake = reinterpret_cast<char*>(align256(top) + 256);
  ChainBwdSet tmp;
  tmp.need_t = S->need_t;
  tmp.need_gt = S->need_gt;
  size_t run_c = 0, query_c = 0;
  rc = plan_chain_composed(op1, op2, tg, ta, tb, tc, grad_a, grad_b, grad_c, nt, szt, numel_t,
                           fake, &tmp, &run_c, &query_c);
  if (rc) return rc;
  // The query covers the route these arguments select (for the fused route
  // whatever pointer alignment; a later call whose pointers select the
  // composed route instead may need more and is refused before launching).
  S->ws_query = S->fused ? fused_q : query_c;
  if (!S->fused) {
    if (workspace) {
      rc = plan_chain_composed(op1, op2, tg, ta, tb, tc, grad_a, grad_b, grad_c, nt, szt, numel_t,
                               static_cast<char*>(workspace), S, &S->ws_run, &query_c);
      if (rc) return rc;
    } else {
      S->ws_run = run_c;
    }
  }
  return ZR_OK;
}

int launch_fwd_set(const FwdSet& S, int op, cudaStream_t st, bool dry) {
  if (S.empty) return ZR_OK;
  if (S.tr) return cuda_status(launch_fwd_tr(op, S.tp, st, dry));
  if (S.sabf) return cuda_status(launch_fwd_sabf(op, S.sp_rpt, S.sp, st, dry));
  return cuda_status(launch_fwd(op, S.eb, st, dry));
}

int launch_chain_set(const ChainBwdSet& S, int op1, int op2, void* workspace, cudaStream_t st,
                     bool dry) {
  if (S.fused) {
    ChainBuild cb = S.cb;
    char* ws = static_cast<char*>(workspace);
    cb.plan.r.partial = reinterpret_cast<float*>(ws);
    cb.comb_b.partial = cb.plan.r.partial;
    cb.plan.c_partial = reinterpret_cast<float*>(ws + S.off_c);
    cb.comb_c.partial = cb.plan.c_partial;
    return cuda_status(launch_chain_bwd(op1, op2, cb, st, dry));
  }
  char* p = static_cast<char*>(workspace) + S.off_p;
  int rc;
  if (S.need_t) {
    rc = launch_fwd_set(S.tf, op1, st, dry);
    if (rc) return rc;
  }
  if (!S.b2.nothing) {
    rc = launch_bwd_set(S.b2, op2, p, st, dry);
    if (rc) return rc;
  }
  if (S.need_gt && !S.b1.nothing) return launch_bwd_set(S.b1, op1, p, st, dry);
  return ZR_OK;
}

std::string describe_chain_set(const ChainBwdSet& S) {
  std::string s;
  if (S.nothing || S.empty) return "{\"route\":\"none\"}";
  if (S.fused) {
    s = "{\"route\":\"fused\",\"plans\":[" + describe_chain(S.cb) + "]";
  } else {
    s = "{\"route\":\"composed\",\"need_t\":" + std::to_string(S.need_t ? 1 : 0) +
        ",\"need_gt\":" + std::to_string(S.need_gt ? 1 : 0);
  }
  return s + ",\"ws_run\":" + std::to_string(S.ws_run) + ",\"ws_query\":" +
         std::to_string(S.ws_query) + "}";
}

}  // namespace
}  // namespace zr

extern "C" {

int zr_chain_fwd(zr_op op1, zr_op op2, zr_tensor a, zr_tensor b, zr_tensor c, float* out,
                 const int64_t* out_strides, zr_stream_t stream) {
  ChainFwdSet S;
  int rc = plan_chain_fwd(op1, op2, a, b, c, out, out_strides, &S);
  if (rc) return rc;
  if (S.empty) return ZR_OK;
  for (const void* p : {static_cast<const void*>(S.a.ptr), static_cast<const void*>(S.b.ptr),
                        static_cast<const void*>(S.c.ptr), static_cast<const void*>(out)}) {
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  return cuda_status(
      launch_chain_fwd(op1, op2, S.c_one, S.eb, reinterpret_cast<cudaStream_t>(stream)));
}

int zr_chain_bwd(zr_op op1, zr_op op2, zr_tensor grad_out, zr_tensor a, zr_tensor b, zr_tensor c,
                 float* grad_a, float* grad_b, float* grad_c, void* workspace,
                 size_t* workspace_bytes, zr_stream_t stream) {
  if (!workspace_bytes) return ZR_ERR_NULL;
  ChainBwdSet S;
  int rc = plan_chain_bwd(op1, op2, grad_out, a, b, c, grad_a, grad_b, grad_c, workspace, &S);
  if (rc) return rc;
  if (workspace == nullptr) {
    *workspace_bytes = S.ws_query;
    return ZR_OK;
  }
  if (S.nothing) return ZR_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S.empty) {
    for (int w = 0; w < 3; ++w) {
      if (!S.zero_ptr[w]) continue;
      rc = check_device_ptr(S.zero_ptr[w]);
      if (rc) return rc;
    }
    for (int w = 0; w < 3; ++w)
      if (S.zero_ptr[w] && cudaMemsetAsync(S.zero_ptr[w], 0, S.zero_bytes[w], st) != cudaSuccess)
        return ZR_ERR_CUDA;
    return ZR_OK;
  }
  if (S.ws_run > 0) {
    if (*workspace_bytes < S.ws_run) return ZR_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return ZR_ERR_WORKSPACE;
  }
  for (const void* p : {static_cast<const void*>(S.g.ptr), static_cast<const void*>(S.a.ptr),
                        static_cast<const void*>(S.b.ptr), static_cast<const void*>(S.c.ptr),
                        static_cast<const void*>(grad_a), static_cast<const void*>(grad_b),
                        static_cast<const void*>(grad_c),
                        S.ws_run > 0 ? static_cast<const void*>(workspace) : nullptr}) {
    if (!p) continue;
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  return launch_chain_set(S, op1, op2, workspace, st, false);
}

int zr_test_describe_chain_bwd(zr_op op1, zr_op op2, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                               zr_tensor c, const float* grad_a, const float* grad_b,
                               const float* grad_c, char* buf, size_t len) {
  ChainBwdSet S;
  const int rc = plan_chain_bwd(op1, op2, grad_out, a, b, c, const_cast<float*>(grad_a),
                                const_cast<float*>(grad_b), const_cast<float*>(grad_c), nullptr,
                                &S);
  if (rc) return rc;
  return copy_json(describe_chain_set(S), buf, len);
}

int zr_test_dry_run_chain_bwd(zr_op op1, zr_op op2, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                              zr_tensor c, const float* grad_a, const float* grad_b,
                              const float* grad_c) {
  // A fake workspace far above any operand address the host tests use.
  void* ws = reinterpret_cast<void*>(uintptr_t(1) << 46);
  ChainBwdSet S;
  const int rc = plan_chain_bwd(op1, op2, grad_out, a, b, c, const_cast<float*>(grad_a),
                                const_cast<float*>(grad_b), const_cast<float*>(grad_c), ws, &S);
  if (rc || S.nothing || S.empty) return rc;
  return launch_chain_set(S, op1, op2, ws, nullptr, true);
}

}  // extern "C"

// ------------------------------------------------------------------ backward with gradient layouts
//
// zr_binary_bwd_ex: each gradient may be strided and may be accumulated
// into (AccumulateGrad, Autograd page, section 反向传播: when the gradient
// slot already holds a value, the new gradient is added in place).  A dense,
// written gradient is written by the backward kernels themselves.  A strided
// or accumulated one is computed densely into the workspace and then copied
// into its layout, or added to it (the elementwise add, in place: old +
// staged, one binary32 addition), by one more elementwise pass; the backward
// kernels themselves only ever store.

namespace zr {
namespace {

struct BwdExSet {
  BwdSet S;
  float* user[2] = {nullptr, nullptr};
  bool stage[2] = {false, false};
  bool acc[2] = {false, false};
  TDesc gd[2];
  EwBuild copy[2];          // staged -> caller's layout: a copy, or (acc) old + staged
  size_t off_stage[2] = {0, 0};
  size_t off_ws = 0;
  size_t ws_run = 0, ws_query = 0;
};

int plan_bwd_ex(int op, const zr_tensor& tg, const zr_tensor& ta, const zr_tensor& tb,
                const zr_grad& ga, const zr_grad& gb, void* workspace, BwdExSet* E) {
  const zr_grad* gs[2] = {&ga, &gb};
  const zr_tensor* ins[2] = {&ta, &tb};
  TDesc in_desc[2], g_desc;
  int rc = read_tensor(tg, &g_desc);
  if (rc) return rc;
  for (int w = 0; w < 2; ++w) {
    rc = read_tensor(*ins[w], &in_desc[w]);
    if (rc) return rc;
    E->user[w] = gs[w]->data;
    E->acc[w] = gs[w]->data && gs[w]->accumulate != 0;
    if (!gs[w]->data) continue;
    const zr_tensor t{gs[w]->data, ins[w]->ndim, ins[w]->sizes, gs[w]->strides};
    rc = read_tensor(t, &E->gd[w]);
    if (rc) return rc;
    if (!non_overlapping(E->gd[w])) return ZR_ERR_LAYOUT;
    E->stage[w] = !dense_layout(E->gd[w]) || E->acc[w];
  }
  // A staged (strided) gradient is checked here against everything else;
  // dense ones are checked by the backward's own plan.
  for (int w = 0; w < 2; ++w) {
    if (!E->stage[w]) continue;
    const Span sp = span_of(E->gd[w].ptr, E->gd[w].extent);
    if (E->user[1 - w] && overlaps(sp, span_of(E->gd[1 - w].ptr, E->gd[1 - w].extent)))
      return ZR_ERR_LAYOUT;
    for (const TDesc* x : {&g_desc, &in_desc[0], &in_desc[1]})
      if (overlaps(sp, span_of(x->ptr, x->extent))) return ZR_ERR_LAYOUT;
  }
  // Workspace: [staged grad_a][staged grad_b][the backward's partials].
  size_t off = 0;
  for (int w = 0; w < 2; ++w) {
    E->off_stage[w] = off;
    if (E->stage[w]) off += align256(size_t(E->gd[w].numel) * 4);
  }
  E->off_ws = off;
  char* base = static_cast<char*>(workspace);
  if (!base) {
    // Query: staging placed above every operand, so no layout check trips.
    uintptr_t top = 0;
    for (const TDesc* x : {&g_desc, &in_desc[0], &in_desc[1], &E->gd[0], &E->gd[1]})
      top = std::max(top, span_of(x->ptr, x->extent).hi);
    base = reinterpret_cast<char*>(align256(top) + 256);
  }
  float* pg[2];
  for (int w = 0; w < 2; ++w)
    pg[w] = E->stage[w] ? reinterpret_cast<float*>(base + E->off_stage[w]) : E->user[w];
  rc = plan_bwd(op, tg, ta, tb, pg[0], pg[1], &E->S);
  if (rc) return rc;
  BwdSet& S = E->S;
  // Move each staged gradient into its layout: copy it, or add it to the old
  // values in place (slot 0: the old values in the caller's layout; slot 1:
  // the staged gradient, dense; the output aliases slot 0 exactly).
  for (int w = 0; w < 2; ++w) {
    if (!E->stage[w] || E->gd[w].numel == 0) continue;
    const TDesc& x = E->gd[w];
    const bool acc = E->acc[w];
    int64_t st[kProbSlots][kMaxDims] = {};
    int64_t dense[kMaxDims];
    contiguous_strides(x.nd, x.size, dense);
    for (int d = 0; d < x.nd; ++d) {
      const int64_t sd = x.size[d] == 1 ? 0 : dense[d];
      const int64_t su = x.size[d] == 1 ? 0 : x.stride[d];
      st[0][d] = acc ? su : sd;
      st[1][d] = acc ? sd : 0;
      st[kSlotOut][d] = su;
    }
    Prob P;
    const uint32_t rmask = acc ? 3u : 1u;
    rc = coalesce(x.nd, x.size, st, rmask | (1u << kSlotOut), kSlotOut, &P);
    if (rc) return rc;
    const float* in[3] = {acc ? E->user[w] : pg[w], acc ? pg[w] : nullptr, nullptr};
    float* outs[2] = {E->user[w], nullptr};
    rc = build_ew(P, in, outs, rmask, rmask, acc ? kOccEwFwd : kOccEwCopy, &E->copy[w]);
    if (rc) return rc;
  }
  E->ws_run = E->off_ws + S.ws_run;
  E->ws_query = E->off_ws + S.ws_query;
  return ZR_OK;
}

}  // namespace
}  // namespace zr

extern "C" {

int zr_binary_bwd_ex(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b, zr_grad grad_a,
                     zr_grad grad_b, void* workspace, size_t* workspace_bytes,
                     zr_stream_t stream) {
  if (!workspace_bytes) return ZR_ERR_NULL;
  BwdExSet E;
  // Plan once to size the workspace; at run time plan again on it.
  int rc = plan_bwd_ex(op, grad_out, a, b, grad_a, grad_b, nullptr, &E);
  if (rc) return rc;
  if (workspace == nullptr) {
    *workspace_bytes = E.ws_query;
    return ZR_OK;
  }
  if (E.S.nothing) return ZR_OK;
  if (E.ws_run > 0) {
    if (*workspace_bytes < E.ws_run) return ZR_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return ZR_ERR_WORKSPACE;
  }
  BwdExSet R;
  rc = plan_bwd_ex(op, grad_out, a, b, grad_a, grad_b, workspace, &R);
  if (rc) return rc;
  if (*workspace_bytes < R.ws_run) return ZR_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const BwdSet& S = R.S;
  const bool ra = (grad_a.data && needs_a(op, 0)) || (grad_b.data && needs_a(op, 1));
  const bool rb = (grad_a.data && needs_b(op, 0)) || (grad_b.data && needs_b(op, 1));
  const void* ptrs[6] = {S.g.ptr,
                         ra ? static_cast<const void*>(S.a.ptr) : nullptr,
                         rb ? static_cast<const void*>(S.b.ptr) : nullptr,
                         grad_a.data,
                         grad_b.data,
                         R.ws_run > 0 ? workspace : nullptr};
  for (const void* p : ptrs) {
    if (!p) continue;
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  if (S.empty) {
    // Nothing to add: an accumulated gradient keeps its values; a written
    // one becomes zero (staged: a zeroed staging buffer copied into place).
    for (int w = 0; w < 2; ++w) {
      if (!S.zero_ptr[w] || R.acc[w]) continue;
      if (cudaMemsetAsync(S.zero_ptr[w], 0, S.zero_bytes[w], st) != cudaSuccess) return ZR_ERR_CUDA;
      if (R.stage[w]) {
        rc = cuda_status(launch_copy(R.copy[w], st));  // a written (not accumulated) gradient
        if (rc) return rc;
      }
    }
    return ZR_OK;
  }
  rc = launch_bwd_set(S, op, static_cast<char*>(workspace) + R.off_ws, st, false);
  if (rc) return rc;
  for (int w = 0; w < 2; ++w) {
    if (!R.stage[w] || R.gd[w].numel == 0) continue;
    rc = cuda_status(R.acc[w] ? launch_fwd(OP_ADD, R.copy[w], st) : launch_copy(R.copy[w], st));
    if (rc) return rc;
  }
  return ZR_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ unary ops
//
// GPU page, section 逐元素运算: GeLU and gradient scaling are elementwise
// (each output element from the input element at the same position).  One
// elementwise pass over x's (or grad_out's) layout; any strides, in place
// allowed with the same layout.

namespace zr {
namespace {

struct UnarySet {
  int es = 4;  // bytes per stored element: 4 float, 2 bfloat16
  bool empty = false;
  EwBuild eb;
  TDesc x, g, out;
};

// in0: x (forward) or grad_out (backward); in1: x for GeLU's backward.
int plan_unary(int uop, float alpha, const zr_tensor& t0, const zr_tensor* t1, float* out,
               const int64_t* out_strides, UnarySet* S) {
  if (uop != UN_SCALE && uop != UN_GELU) return ZR_ERR_NULL;
  int rc = read_tensor(t0, &S->g);
  if (rc) return rc;
  const bool two = t1 != nullptr;
  if (two) {
    rc = read_tensor(*t1, &S->x);
    if (rc) return rc;
    if (S->x.nd != S->g.nd) return ZR_ERR_SHAPE;
    for (int d = 0; d < S->g.nd; ++d)
      if (S->x.size[d] != S->g.size[d]) return ZR_ERR_SHAPE;
  }
  const int n = S->g.nd;
  zr_tensor to{out, n, S->g.size, out_strides};
  rc = read_tensor(to, &S->out);
  if (rc) return rc;
  if (S->out.numel == 0) {
    S->empty = true;
    return ZR_OK;
  }
  if (!S->g.ptr || !out || (two && !S->x.ptr)) return ZR_ERR_NULL;
  if (!non_overlapping(S->out)) return ZR_ERR_LAYOUT;
  const Span so = span_of(out, S->out.extent, S->es);
  if (overlaps(so, span_of(S->g.ptr, S->g.extent, S->es)) && !same_layout(S->g, S->out))
    return ZR_ERR_LAYOUT;
  if (two && overlaps(so, span_of(S->x.ptr, S->x.extent, S->es)) && !same_layout(S->x, S->out))
    return ZR_ERR_LAYOUT;
  int64_t st[kProbSlots][kMaxDims] = {};
  for (int d = 0; d < n; ++d) {
    const bool one = S->g.size[d] == 1;
    st[0][d] = one ? 0 : S->g.stride[d];
    st[1][d] = (one || !two) ? 0 : S->x.stride[d];
    st[kSlotOut][d] = one ? 0 : S->out.stride[d];
  }
  Prob P;
  const uint32_t rmask = two ? 3u : 1u;
  rc = coalesce(n, S->g.size, st, rmask | (1u << kSlotOut), kSlotOut, &P);
  if (rc) return rc;
  P.es = S->es;
  const float* in[3] = {S->g.ptr, two ? S->x.ptr : nullptr, nullptr};
  float* outs[2] = {out, nullptr};
  rc = build_ew(P, in, outs, rmask, rmask, kOccEwFwd, &S->eb);
  if (rc) return rc;
  S->eb.plan.alpha = alpha;
  // bfloat16 GeLU over a flat layout large enough to amortise the table:
  // one CTA per SM (fewer if there are fewer passes of the kernel's loads).
  EwPlan& ep = S->eb.plan;
  if (uop == UN_GELU && S->es == 2 && ep.flat &&
      uint64_t(ep.nitems) * uint64_t(S->eb.vec) >= kGeluTabMinElems) {
    const uint64_t pass = uint64_t(two ? kGeluTabUnrollBwd : kGeluTabUnrollFwd) * kGeluTabThreads;
    S->eb.gelu_tab = true;
    ep.n_cta = uint32_t(std::min<uint64_t>(kSms, (uint64_t(ep.nitems) + pass - 1) / pass));
  }
  return ZR_OK;
}

}  // namespace
}  // namespace zr

extern "C" {

int zr_unary_fwd(zr_unary op, float alpha, zr_tensor x, float* out, const int64_t* out_strides,
                 zr_stream_t stream) {
  return zr_unary_fwd_t(ZR_F32, op, alpha, x, out, out_strides, stream);
}

int zr_unary_fwd_t(zr_dtype dtype, zr_unary op, float alpha, zr_tensor x, void* out_v,
                   const int64_t* out_strides, zr_stream_t stream) {
  if (dtype != ZR_F32 && dtype != ZR_BF16) return ZR_ERR_DTYPE;
  float* out = static_cast<float*>(out_v);
  UnarySet S;
  S.es = dtype == ZR_BF16 ? 2 : 4;
  int rc = plan_unary(op, alpha, x, nullptr, out, out_strides, &S);
  if (rc || S.empty) return rc;
  if (trace_on()) trace("zr_unary_fwd", describe_ew(S.eb));
  for (const void* p : {static_cast<const void*>(S.g.ptr), static_cast<const void*>(out)}) {
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  return cuda_status(launch_unary_fwd(op, S.eb, reinterpret_cast<cudaStream_t>(stream)));
}

int zr_unary_bwd(zr_unary op, float alpha, zr_tensor grad_out, zr_tensor x, float* grad_x,
                 const int64_t* grad_x_strides, zr_stream_t stream) {
  return zr_unary_bwd_t(ZR_F32, op, alpha, grad_out, x, grad_x, grad_x_strides, stream);
}

int zr_unary_bwd_t(zr_dtype dtype, zr_unary op, float alpha, zr_tensor grad_out, zr_tensor x,
                   void* grad_x_v, const int64_t* grad_x_strides, zr_stream_t stream) {
  if (dtype != ZR_F32 && dtype != ZR_BF16) return ZR_ERR_DTYPE;
  float* grad_x = static_cast<float*>(grad_x_v);
  UnarySet S;
  S.es = dtype == ZR_BF16 ? 2 : 4;
  // scale's backward does not read x (its sizes must still match grad_out).
  int rc = plan_unary(op, alpha, grad_out, op == UN_GELU ? &x : nullptr, grad_x, grad_x_strides,
                      &S);
  if (rc || S.empty) return rc;
  if (trace_on()) trace("zr_unary_bwd", describe_ew(S.eb));
  if (op != UN_GELU) {
    if (x.ndim != grad_out.ndim || (x.ndim > 0 && !x.sizes)) return ZR_ERR_SHAPE;
    for (int d = 0; d < x.ndim; ++d)
      if (x.sizes[d] != S.g.size[d]) return ZR_ERR_SHAPE;
  }
  for (const void* p : {static_cast<const void*>(S.g.ptr),
                        op == UN_GELU ? static_cast<const void*>(S.x.ptr) : nullptr,
                        static_cast<const void*>(grad_x)}) {
    if (!p) continue;
    rc = check_device_ptr(p);
    if (rc) return rc;
  }
  return cuda_status(launch_unary_bwd(op, S.eb, reinterpret_cast<cudaStream_t>(stream)));
}

int zr_test_describe_unary_t(zr_dtype dtype, zr_unary op, zr_tensor in0, const zr_tensor* x,
                             const void* out, const int64_t* out_strides, char* buf, size_t len) {
  if (dtype != ZR_F32 && dtype != ZR_BF16) return ZR_ERR_DTYPE;
  UnarySet S;
  S.es = dtype == ZR_BF16 ? 2 : 4;
  const int rc = plan_unary(op, 1.f, in0, x, static_cast<float*>(const_cast<void*>(out)),
                            out_strides, &S);
  if (rc) return rc;
  return copy_json(S.empty ? std::string("{\"kernel\":\"none\"}") : describe_ew(S.eb), buf, len);
}

}  // extern "C"
