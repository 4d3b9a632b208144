// zr_kernels.cuh — CUDA kernels (sm_103a) for broadcasting elementwise
// binary ops, their fused backward and deterministic sum-to-shape.
//
// Arithmetic is explicit: __fadd_rn/__fsub_rn/__fmul_rn/__fdiv_rn are IEEE
// binary32 operations with round-to-nearest-even that the compiler never
// contracts into FMAs, and the library is built with -ftz=false, so a
// forward element is exactly the one IEEE operation the Zero book's
// Operator page (section 逐元素算子) names for it.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include "zr_internal.h"
#include "zr_launch.h"

namespace zr {

// ---------------------------------------------------------------- arithmetic

// x / y correctly rounded to binary32 (round to nearest even) for x and y
// that bfloat16 can hold (8-bit significands), without the general divide:
// an approximate quotient and one correction with the exact residual, as in
// P. W. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990:
//   r = approx 1/y,  q0 = x * r,  e = x - y * q0 (one FMA),  q = q0 + e * r.
// Valid when div_fast_ok: both exponents in [-60, 60], so nothing
// overflows, underflows or turns subnormal, and q0 + e * r is within 2^-43
// of x / y (relative).  For 8-bit significands A, B the quotient is never
// exactly halfway between two binary32 numbers (A = (2m + 1) B with 2m + 1
// odd and above 2^24 is impossible) and otherwise at least 2^-33 (relative)
// away from every halfway point, so the FMA's one rounding gives RN(x / y).
// Every pair of bfloat16 values is checked against the IEEE divide by a GPU
// test.
__device__ __forceinline__ float div_fast(float x, float y) {
  float r;  // y is normal here, so the flush-to-zero form is exact enough
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-y, q0, x);
  return __fmaf_rn(e, r, q0);
}
// 2^-60 <= |v| < 2^61 (false for zeros, subnormals, infinities and NaNs).
__device__ __forceinline__ bool div_fast_range(float v) {
  const float m = fabsf(v);
  return (m >= 0x1p-60f) & (m < 0x1p61f);
}
__device__ __forceinline__ bool div_fast_ok(float x, float y) {
  return div_fast_range(x) & div_fast_range(y);
}

// Division by a power of two as a multiplication: when d = +-2^k and 1/d are
// both normal binary32 numbers (k in [-126, 126]), x / d and x * (1/d) are
// the same real number for every x, so their single roundings agree bit for
// bit, zeros, infinities, NaNs and results in the subnormal range included.
// Sets *r = 1/d (exact) and returns true for such d.
__device__ __forceinline__ bool pow2_reciprocal(float d, float* r) {
  const uint32_t u = __float_as_uint(d);
  const uint32_t e = (u >> 23) & 0xFFu;
  if ((u & 0x7FFFFFu) != 0u || e < 1u || e > 253u) return false;
  *r = __uint_as_float((u & 0x80000000u) | ((254u - e) << 23));
  return true;
}

template <int OP>
__device__ __forceinline__ float fwd_op(float x, float y) {
  if (OP == OP_ADD) return __fadd_rn(x, y);
  if (OP == OP_SUB) return __fsub_rn(x, y);
  if (OP == OP_MUL) return __fmul_rn(x, y);
  return __fdiv_rn(x, y);
}

// Local gradient terms.  add (g, g) — GPU page, section OpAdd; mul (g*b, g*a)
// — Operator page, section 逐元素算子; sub (g, -g) and div (g/b, -g*a/b^2) by
// calculus (the pages do not write them out).  Every single-operation term
// (all but div's grad_b) is the exact IEEE result.
template <int OP>
__device__ __forceinline__ float term_a(float g, float a, float b) {
  (void)a;
  if (OP == OP_ADD || OP == OP_SUB) return g;
  if (OP == OP_MUL) return __fmul_rn(g, b);
  return __fdiv_rn(g, b);
}
template <int OP>
__device__ __forceinline__ float term_b(float g, float a, float b) {
  if (OP == OP_ADD) return g;
  if (OP == OP_SUB) return -g;
  if (OP == OP_MUL) return __fmul_rn(g, a);
  return -__fmul_rn(__fdiv_rn(g, b), __fdiv_rn(a, b));
}

// Which inputs a gradient reads.  WHICH: 0 = grad_a, 1 = grad_b.
template <int OP, int WHICH>
struct Needs {
  static constexpr bool a = (WHICH == 1) && (OP == OP_MUL || OP == OP_DIV);
  static constexpr bool b = (WHICH == 0 && (OP == OP_MUL || OP == OP_DIV)) ||
                            (WHICH == 1 && OP == OP_DIV);
};

// Compensated (Kahan) summation: error <= (2u + O(n u^2)) * sum|x_i| whatever
// the number of terms (N. J. Higham, "Accuracy and Stability of Numerical
// Algorithms", 2nd ed., section 4.3).  Explicit _rn intrinsics keep the
// compiler from reassociating or contracting the compensation away.
// Programmatic dependent launch.  Every kernel starts with pdl_trigger()
// (the next kernel in the stream may now be scheduled; it runs only its own
// parameter-only setup before its pdl_wait()), computes what depends on its
// parameters alone (index decompositions, shared-memory offset tables), and
// calls pdl_wait() before its first access to global memory: that returns
// once the grids before it in the stream have completed and their writes are
// visible (at once when the launch did not ask for programmatic
// serialization).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Thread-block clusters.  cluster_sync(): every thread of every CTA of the
// cluster arrives (release: this CTA's shared-memory writes become visible
// to the cluster) and waits for all (acquire).  All CTAs of a cluster are
// resident together by construction, so the wait always ends.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// The float at the same shared-memory offset as `local` in CTA `rank` of
// this cluster (distributed shared memory).
__device__ __forceinline__ float ld_cluster(const float* local, uint32_t rank) {
  const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(la), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// cp.async: 16-byte copies from global to shared memory that complete in the
// background; a thread waits for its own groups of copies with
// cp_async_wait<N>() (at most N most recent groups still in flight), after
// which the copied bytes are visible to that thread.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

struct Kahan {
  float s, c;
  __device__ __forceinline__ void init() { s = 0.f; c = 0.f; }
  __device__ __forceinline__ void add(float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
  // Adds the exact product u*v: the FMA forms u*v - c with one rounding, so
  // the summed term carries no product rounding error.
  __device__ __forceinline__ void add_prod(float u, float v) {
    const float y = __fmaf_rn(u, v, -c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
};

// ---------------------------------------------------------------- loads/stores

template <int VEC>
struct Vec { float v[VEC]; };

// Quotients x / y of VEC pairs of bfloat16 values: div_fast for all when
// every pair is in its range, else the IEEE divide for all (one branch per
// vector, so the VEC independent reciprocal-and-correction chains
// interleave).  Bit-identical to __fdiv_rn on every pair either way.
template <int VEC>
__device__ __forceinline__ void quot_short(const Vec<VEC>& x, const Vec<VEC>& y, Vec<VEC>& q) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < VEC; ++i) ok = ok & div_fast_ok(x.v[i], y.v[i]);
  if (ok) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) q.v[i] = div_fast(x.v[i], y.v[i]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) q.v[i] = __fdiv_rn(x.v[i], y.v[i]);
  }
}

// Quotients x / y of VEC pairs of bfloat16 values whose results are stored
// as bfloat16: q = x * (approximate 1/y), one rounding.  Its relative error is
// below 2^-22, and x / y is never exactly halfway between two bfloat16
// numbers and otherwise more than 2^-18 (relative) away from every halfway
// point: a halfway point is N 2^t with N odd, 2^8 < N < 2^9, and x = A 2^i,
// y = B 2^j with A, B below 2^8 make x - N 2^t y a nonzero multiple of
// 2^min(i, t+j) (A = N B odd-part-wise is impossible), so
// |x/y - N 2^t| >= 2^min(i, t+j) / y, relatively at least about
// 1 / (B N) > 2^-17.  So q and x / y round to
// the same bfloat16 number, which is RN(RN(x / y)) by the innocuous double
// rounding of 24 >= 2 * 8 + 2 bits.  Valid when every pair passes
// div_fast_ok (q is then a normal number); otherwise the IEEE divide for all.
template <int VEC>
__device__ __forceinline__ void quot_bf16(const Vec<VEC>& x, const Vec<VEC>& y, Vec<VEC>& q) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < VEC; ++i) ok = ok & div_fast_ok(x.v[i], y.v[i]);
  if (ok) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      float r;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y.v[i]));
      q.v[i] = __fmul_rn(x.v[i], r);
    }
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) q.v[i] = __fdiv_rn(x.v[i], y.v[i]);
  }
}

// Vector forms of the forward and of the dense gradient terms.  SHORT: the
// operands are bfloat16 values and the results are stored as bfloat16: a
// stored quotient takes quot_bf16, a quotient that feeds a product
// quot_short; otherwise (and for the other ops) the scalar forms above,
// element by element.
template <int OP, bool SHORT, int VEC>
__device__ __forceinline__ void fwd_vec(const Vec<VEC>& x, const Vec<VEC>& y, Vec<VEC>& out) {
  if (OP == OP_DIV && SHORT) {
    quot_bf16(x, y, out);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) out.v[i] = fwd_op<OP>(x.v[i], y.v[i]);
  }
}
template <int OP, bool SHORT, int VEC>
__device__ __forceinline__ void term_a_vec(const Vec<VEC>& g, const Vec<VEC>& a, const Vec<VEC>& b,
                                           Vec<VEC>& out) {
  if (OP == OP_DIV && SHORT) {
    quot_bf16(g, b, out);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) out.v[i] = term_a<OP>(g.v[i], a.v[i], b.v[i]);
  }
}
template <int OP, bool SHORT, int VEC>
__device__ __forceinline__ void term_b_vec(const Vec<VEC>& g, const Vec<VEC>& a, const Vec<VEC>& b,
                                           Vec<VEC>& out) {
  if (OP == OP_DIV && SHORT) {
    Vec<VEC> qg, qa;
    quot_short(g, b, qg);
    quot_short(a, b, qa);
#pragma unroll
    for (int i = 0; i < VEC; ++i) out.v[i] = -__fmul_rn(qg.v[i], qa.v[i]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) out.v[i] = term_b<OP>(g.v[i], a.v[i], b.v[i]);
  }
}

// Storage types E: float, or bfloat16 (binary32's upper 16 bits).  Loads
// widen to binary32 exactly; stores round to the storage type once, to
// nearest with ties to even.  All arithmetic is binary32.
__device__ __forceinline__ float ld1(const float* p, bool streaming) {
  return streaming ? __ldcs(p) : __ldg(p);
}
__device__ __forceinline__ float ld1(const __nv_bfloat16* p, bool streaming) {
  const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
  const unsigned short u = streaming ? __ldcs(q) : __ldg(q);
  return __uint_as_float(uint32_t(u) << 16);
}
__device__ __forceinline__ void st1(float* p, float v) { *p = v; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// What a thread holds between issuing a load and using it: the binary32
// values themselves for float storage; for bfloat16 the packed 16-bit
// patterns, two per 32-bit word, so that a 16-byte load of 8 elements takes
// 4 registers (not 8) until the values are used.
template <class E, int VEC>
struct Raw { Vec<VEC> x; };
template <int VEC>
struct Raw<__nv_bfloat16, VEC> { uint32_t w[(VEC + 1) / 2]; };

template <int VEC>
__device__ __forceinline__ Raw<__nv_bfloat16, VEC> load_raw_bf16(const __nv_bfloat16* base,
                                                                  int64_t row_off, int64_t inner,
                                                                  uint32_t c, bool streaming) {
  Raw<__nv_bfloat16, VEC> r;
  const unsigned short* b = reinterpret_cast<const unsigned short*>(base);
  if (inner == 1) {
    const unsigned short* p = b + row_off + c;
    if constexpr (VEC == 8) {
      const uint4 q = streaming ? __ldcs(reinterpret_cast<const uint4*>(p))
                                : __ldg(reinterpret_cast<const uint4*>(p));
      r.w[0] = q.x; r.w[1] = q.y; r.w[2] = q.z; r.w[3] = q.w;
    } else if constexpr (VEC == 4) {
      const uint2 q = streaming ? __ldcs(reinterpret_cast<const uint2*>(p))
                                : __ldg(reinterpret_cast<const uint2*>(p));
      r.w[0] = q.x; r.w[1] = q.y;
    } else {
      r.w[0] = streaming ? __ldcs(p) : __ldg(p);
    }
  } else if (inner == 0) {
    const uint32_t u = __ldg(b + row_off);
#pragma unroll
    for (int i = 0; i < (VEC + 1) / 2; ++i) r.w[i] = u | (u << 16);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const uint32_t u = __ldg(b + row_off + int64_t(c + i) * inner);
      if (i & 1) r.w[i / 2] |= u << 16;
      else r.w[i / 2] = u;
    }
  }
  return r;
}

template <int VEC>
__device__ __forceinline__ Vec<VEC> unpack_bf16(const Raw<__nv_bfloat16, VEC>& r) {
  Vec<VEC> v;
#pragma unroll
  for (int i = 0; i < VEC; ++i)
    v.v[i] = __uint_as_float((i & 1) ? (r.w[i / 2] & 0xFFFF0000u) : (r.w[i / 2] << 16));
  return v;
}

// A 16-byte vector staged in shared memory as the register form a load
// would have produced (4 floats, or 8 bfloat16 kept packed).
template <class E, int VEC>
__device__ __forceinline__ Raw<E, VEC> raw_from_u4(const uint4& q) {
  static_assert(VEC * sizeof(E) == 16, "16-byte vectors only");
  Raw<E, VEC> r;
  if constexpr (sizeof(E) == 2) {
    r.w[0] = q.x; r.w[1] = q.y; r.w[2] = q.z; r.w[3] = q.w;
  } else {
    r.x.v[0] = __uint_as_float(q.x); r.x.v[1] = __uint_as_float(q.y);
    r.x.v[2] = __uint_as_float(q.z); r.x.v[3] = __uint_as_float(q.w);
  }
  return r;
}

// Load VEC consecutive columns of one operand in one row.  inner == 1:
// contiguous (one 16-byte load of 4 floats or one 8-byte load of 4 bf16 when
// VEC == 4; the planner guarantees alignment); inner == 0: the column is
// broadcast, one load; otherwise a strided gather.
template <int VEC, class E>
__device__ __forceinline__ Vec<VEC> load_cols(const E* __restrict__ base, int64_t row_off,
                                              int64_t inner, uint32_t c, bool streaming) {
  if constexpr (sizeof(E) == 2) {
    return unpack_bf16<VEC>(load_raw_bf16<VEC>(base, row_off, inner, c, streaming));
  }
  Vec<VEC> r;
  if (inner == 1) {
    const E* p = base + row_off + c;
    if constexpr (VEC % 4 == 0) {
#pragma unroll
      for (int k = 0; k < VEC; k += 4) {
        const float4 q = streaming ? __ldcs(reinterpret_cast<const float4*>(p + k))
                                   : __ldg(reinterpret_cast<const float4*>(p + k));
        r.v[k] = q.x; r.v[k + 1] = q.y; r.v[k + 2] = q.z; r.v[k + 3] = q.w;
      }
    } else {
      static_assert(VEC == 1, "vector width");
      r.v[0] = ld1(p, streaming);
    }
  } else if (inner == 0) {
    const float s = ld1(base + row_off, false);
#pragma unroll
    for (int i = 0; i < VEC; ++i) r.v[i] = s;
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) r.v[i] = ld1(base + row_off + int64_t(c + i) * inner, false);
  }
  return r;
}

template <int VEC, class E>
__device__ __forceinline__ Raw<E, VEC> load_raw(const E* __restrict__ base, int64_t row_off,
                                                int64_t inner, uint32_t c, bool streaming) {
  if constexpr (sizeof(E) == 2) {
    return load_raw_bf16<VEC>(base, row_off, inner, c, streaming);
  } else {
    Raw<E, VEC> r;
    r.x = load_cols<VEC>(base, row_off, inner, c, streaming);
    return r;
  }
}
template <int VEC, class E>
__device__ __forceinline__ Vec<VEC> unpack(const Raw<E, VEC>& r) {
  if constexpr (sizeof(E) == 2) return unpack_bf16<VEC>(r);
  else return r.x;
}

template <int VEC, class E>
__device__ __forceinline__ void store_cols(E* __restrict__ base, int64_t row_off, int64_t inner,
                                           uint32_t c, const Vec<VEC>& x) {
  if (inner == 1) {
    E* p = base + row_off + c;
    if constexpr (sizeof(E) == 4 && VEC % 4 == 0) {
      // 16-byte stores of 4 floats (binary32 partial slots of an 8-wide
      // bfloat16 reduction take two).
#pragma unroll
      for (int k = 0; k < VEC; k += 4)
        *reinterpret_cast<float4*>(p + k) = make_float4(x.v[k], x.v[k + 1], x.v[k + 2], x.v[k + 3]);
    } else if constexpr (sizeof(E) == 2 && VEC == 8) {
      *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(x.v[0], x.v[1]), pack_bf16x2(x.v[2], x.v[3]),
                                                pack_bf16x2(x.v[4], x.v[5]), pack_bf16x2(x.v[6], x.v[7]));
    } else if constexpr (sizeof(E) == 2 && VEC == 4) {
      *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(x.v[0], x.v[1]), pack_bf16x2(x.v[2], x.v[3]));
    } else {
      static_assert(VEC == 1, "vector width");
      st1(p, x.v[0]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) st1(base + row_off + int64_t(c + i) * inner, x.v[i]);
  }
}

// ---------------------------------------------------------------- functors

// Forward: out = a op b.  SHORT: operands are bfloat16 values (fwd_vec's
// division for stored bfloat16 results).
// B_ONE: b has one element, read once per thread (its reciprocal and range
// check are then loop-invariant).
template <int OP, bool SHORT = false, bool B_ONE = false>
struct FwdF {
  static constexpr bool kR1 = true, kR2 = false;  // slot 0 = a, slot 1 = b
  static constexpr bool kUniform1 = B_ONE;
  static constexpr int kMinBlocks = kOccEwFwd;  // CTAs per SM the register budget targets
  static constexpr int kMinBlocksWide = kOccEwFwd;
  template <int VEC>
  __device__ __forceinline__ void operator()(const Vec<VEC> (&x)[3], Vec<VEC> (&y)[2], float) const {
    if (OP == OP_DIV && B_ONE) {
      // One divisor for every element: a power of two divides by one exact
      // multiplication (pow2_reciprocal; the check depends only on the
      // divisor, so it is made once per thread).
      float r;
      if (pow2_reciprocal(x[1].v[0], &r)) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) y[0].v[i] = __fmul_rn(x[0].v[i], r);
        return;
      }
    }
    fwd_vec<OP, SHORT>(x[0], x[1], y[0]);
  }
};

// Backward with no reduction: grad_a and/or grad_b elementwise.
// Inputs: slot 0 = g, 1 = a, 2 = b.  WANT: bit 0 grad_a, bit 1 grad_b.
template <int OP, int WANT, bool SHORT = false>
struct BwdDirectF {
  static constexpr bool kR1 = ((WANT & 1) && Needs<OP, 0>::a) || ((WANT & 2) && Needs<OP, 1>::a);
  static constexpr bool kR2 = ((WANT & 1) && Needs<OP, 0>::b) || ((WANT & 2) && Needs<OP, 1>::b);
  static constexpr int kMinBlocks = kOccEwBwd;
  static constexpr int kMinBlocksWide = (OP == OP_DIV && (WANT & 2)) ? 2 : kOccEwBwd;
  template <int VEC>
  __device__ __forceinline__ void operator()(const Vec<VEC> (&x)[3], Vec<VEC> (&y)[2], float) const {
    if (WANT & 1) term_a_vec<OP, SHORT>(x[0], x[1], x[2], y[0]);
    if (WANT & 2) term_b_vec<OP, SHORT>(x[0], x[1], x[2], y[1]);
  }
};

// Forward of a two-op chain: out = (a op1 b) op2 c, each op one IEEE
// binary32 operation (the intermediate is rounded as the unfused ops would
// store it).  Slots 0, 1, 2 = a, b, c.  C_ONE: c has one element, loaded once
// per thread instead of per item (fewer registers: 4 CTAs per SM).
template <int OP1, int OP2, bool C_ONE>
struct ChainF {
  static constexpr bool kR1 = true, kR2 = true;
  static constexpr bool kUniform2 = C_ONE;
  static constexpr int kMinBlocks = C_ONE ? kOccEwFwd : kOccEwBwd;
  template <int VEC>
  __device__ __forceinline__ void operator()(const Vec<VEC> (&x)[3], Vec<VEC> (&y)[2], float) const {
#pragma unroll
    for (int i = 0; i < VEC; ++i) y[0].v[i] = fwd_op<OP2>(fwd_op<OP1>(x[0].v[i], x[1].v[i]), x[2].v[i]);
  }
};

// Unary elementwise ops (GPU page, section 逐元素运算: GeLU and gradient
// scaling compute each output element from the input element at the same
// position).  scale: alpha * x, one IEEE binary32 multiply.  GeLU: the exact
// x * Phi(x), Phi(x) = erfc(-x / sqrt(2)) / 2 (erfc avoids the cancellation of
// 1 + erf for negative x); its derivative Phi(x) + x * phi(x),
// phi(x) = exp(-x^2 / 2) / sqrt(2 pi).  Slot 0: x (forward) or grad_out
// (backward); slot 1: x (GeLU backward).
//
// GeLU is bound by arithmetic, not memory, so erfc is evaluated with the
// Chebyshev-fitted form of W. H. Press et al., "Numerical Recipes", section
// 6.2 (erfc(z) = t exp(-z^2 + P(t)), t = 1 / (1 + z/2), P of degree 9;
// fractional error below 1.2e-7 for z >= 0, and erfc(-z) = 2 - erfc(z)), with
// the hardware's approximate reciprocal and base-2 exponential
// (exp(v) = 2^(v log2 e)).  Their errors (a few ulp, plus the rounding of
// the exponent's argument, relative |v| u) stay inside the stated bound
// (16 + 2 x^2) * 2^-24 of the exact value.
// Both in their flush-to-zero forms, which skip the subnormal handling: the
// reciprocal's argument is at least 1, and an exponential below 2^-126
// (erfc or phi in their far tails) becomes 0, an absolute change below the
// bound's 2^-120 term.
__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// P(t) of the degree-9 form, highest coefficient first.
#define ZR_ERFC_CHEB_P                                                                          \
  0.17087277f, -0.82215223f, 1.48851587f, -1.13520398f, 0.27886807f, -0.18628806f, 0.09678418f, \
      0.37409196f, 1.00002368f, -1.26551223f
__device__ __forceinline__ float erfc_cheb(float v) {
  constexpr float kP[10] = {ZR_ERFC_CHEB_P};
  const float z = fabsf(v);
  const float t = rcp_approx(__fmaf_rn(0.5f, z, 1.0f));
  float q = kP[0];  // P(t), Horner from the highest coefficient
#pragma unroll
  for (int k = 1; k < 10; ++k) q = __fmaf_rn(q, t, kP[k]);
  const float y = __fmul_rn(t, ex2_approx(__fmul_rn(__fmaf_rn(-z, z, q), 1.44269504088896341f)));
  return v >= 0.f ? y : __fsub_rn(2.0f, y);
}
// erfc for GeLU results stored as bfloat16: the same form with P of degree 5,
// fitted by least squares on Chebyshev nodes of t in [1/8, 1] (z in [0, 14];
// erfc_fit.py beside this file derives these coefficients and measures the
// fit).  Relative error below 1.3e-5 (2^-16.3) with binary32 evaluation:
// far inside bfloat16's half unit of 2^-9, at four fewer multiply-adds.
// P(t) of the degree-5 form, highest coefficient first.
#define ZR_ERFC_SHORT_P                                                          \
  0.22462645173072815f, -0.6965311169624329f, 0.45995479822158813f,              \
      0.2622242867946625f, 1.0161044597625732f, -1.2663732767105103f
__device__ __forceinline__ float erfc_short(float v) {
  constexpr float kP[6] = {ZR_ERFC_SHORT_P};
  const float z = fabsf(v);
  const float t = rcp_approx(__fmaf_rn(0.5f, z, 1.0f));
  float q = kP[0];  // P(t), Horner from the highest coefficient
#pragma unroll
  for (int k = 1; k < 6; ++k) q = __fmaf_rn(q, t, kP[k]);
  const float y = __fmul_rn(t, ex2_approx(__fmul_rn(__fmaf_rn(-z, z, q), 1.44269504088896341f)));
  return v >= 0.f ? y : __fsub_rn(2.0f, y);
}
// Two binary32 lanes in one 64-bit register, for Blackwell's packed FP32
// instructions: add/mul/fma.rn.f32x2 round each lane exactly as the scalar
// __fadd_rn/__fmul_rn/__fmaf_rn do, at one issue slot per pair.  The
// approximate reciprocal and exponential stay scalar (one per lane).
struct F2 {
  unsigned long long v;
};
__device__ __forceinline__ F2 f2_pack(float lo, float hi) {
  F2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ F2 f2_splat(float x) { return f2_pack(x, x); }
__device__ __forceinline__ void f2_unpack(F2 a, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  F2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  F2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
// Sign operations on both lanes' bit patterns (exact, like fabsf and -x).
__device__ __forceinline__ F2 f2_abs(F2 a) { return F2{a.v & 0x7FFFFFFF7FFFFFFFull}; }
__device__ __forceinline__ F2 f2_neg(F2 a) { return F2{a.v ^ 0x8000000080000000ull}; }

// erfc of both lanes: the same operations, in the same order, as erfc_cheb
// (SHORT = false) or erfc_short (SHORT = true), so each lane's result is
// bit-identical to theirs.
template <bool SHORT>
__device__ __forceinline__ F2 erfc2(F2 v) {
  const F2 z = f2_abs(v);
  float d0, d1;
  f2_unpack(f2_fma(f2_splat(0.5f), z, f2_splat(1.0f)), d0, d1);
  const F2 t = f2_pack(rcp_approx(d0), rcp_approx(d1));
  constexpr float kShort[6] = {ZR_ERFC_SHORT_P};
  constexpr float kCheb[10] = {ZR_ERFC_CHEB_P};
  constexpr int kN = SHORT ? 6 : 10;
  F2 q = f2_splat(SHORT ? kShort[0] : kCheb[0]);
#pragma unroll
  for (int k = 1; k < kN; ++k) q = f2_fma(q, t, f2_splat(SHORT ? kShort[k] : kCheb[k]));
  float e0, e1;
  f2_unpack(f2_mul(f2_fma(f2_neg(z), z, q), f2_splat(1.44269504088896341f)), e0, e1);
  const F2 y = f2_mul(t, f2_pack(ex2_approx(e0), ex2_approx(e1)));
  const F2 w = f2_fma(y, f2_splat(-1.0f), f2_splat(2.0f));  // RN(2 - y)
  float v0, v1, y0, y1, w0, w1;
  f2_unpack(v, v0, v1);
  f2_unpack(y, y0, y1);
  f2_unpack(w, w0, w1);
  return f2_pack(v0 >= 0.f ? y0 : w0, v1 >= 0.f ? y1 : w1);
}
// Phi of both lanes, as gelu_cdf.
template <bool SHORT>
__device__ __forceinline__ F2 gelu_cdf2(F2 x) {
  const F2 v = f2_mul(f2_neg(x), f2_splat(0.70710678118654752f));
  return f2_mul(f2_splat(0.5f), erfc2<SHORT>(v));
}

// Phi(x) = erfc(-x / sqrt 2) / 2; SHORT: the result is stored as bfloat16.
template <bool SHORT = false>
__device__ __forceinline__ float gelu_cdf(float x) {
  const float v = __fmul_rn(-x, 0.70710678118654752f);
  return __fmul_rn(0.5f, SHORT ? erfc_short(v) : erfc_cheb(v));
}
template <int UOP, bool SHORT = false>
struct UnaryF {
  static constexpr bool kR1 = false, kR2 = false;
  // GeLU's arithmetic per load is long, so it gains from more resident warps
  // rather than more loads in flight per thread: float GeLU at 5 CTAs per SM
  // (u1 forward 64.2 -> 61.4 us), the 8-wide bfloat16 one at 6 CTAs per SM
  // with 2 items per batch in the flat kernel (u1h forward 45.1 -> 43.1 us);
  // neither spills.
  static constexpr int kMinBlocks = UOP == UN_GELU ? kOccGeluFwd : kOccEwFwd;
  static constexpr int kMinBlocksWide = UOP == UN_GELU ? kOccGeluFwdWide : kOccEwFwd;
  static constexpr int kUnroll = (UOP == UN_GELU && SHORT) ? 2 : 4;
  template <int VEC>
  __device__ __forceinline__ void operator()(const Vec<VEC> (&x)[3], Vec<VEC> (&y)[2], float alpha) const {
    if constexpr (UOP == UN_GELU && VEC % 2 == 0) {
      // Pairs of elements through the packed instructions (same results).
#pragma unroll
      for (int i = 0; i < VEC; i += 2) {
        const F2 v = f2_pack(x[0].v[i], x[0].v[i + 1]);
        f2_unpack(f2_mul(v, gelu_cdf2<SHORT>(v)), y[0].v[i], y[0].v[i + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float v = x[0].v[i];
        y[0].v[i] = UOP == UN_SCALE ? __fmul_rn(alpha, v) : __fmul_rn(v, gelu_cdf<SHORT>(v));
      }
    }
  }
};
template <int UOP, bool SHORT = false>
struct UnaryBwdF {
  static constexpr bool kR1 = UOP == UN_GELU, kR2 = false;
  static constexpr int kMinBlocks = kOccEwFwd;
  // 8-wide bfloat16 GeLU backward (two operand streams) needs 80 registers.
  static constexpr int kMinBlocksWide = UOP == UN_GELU ? kOccEwFwd - 1 : kOccEwFwd;
  template <int VEC>
  __device__ __forceinline__ void operator()(const Vec<VEC> (&x)[3], Vec<VEC> (&y)[2], float alpha) const {
    if constexpr (UOP == UN_GELU && VEC % 2 == 0) {
      // Pairs of elements through the packed instructions (same results).
#pragma unroll
      for (int i = 0; i < VEC; i += 2) {
        const F2 g = f2_pack(x[0].v[i], x[0].v[i + 1]);
        const F2 v = f2_pack(x[1].v[i], x[1].v[i + 1]);
        float a0, a1;
        f2_unpack(f2_mul(f2_mul(f2_splat(-0.72134752044448170f), v), v), a0, a1);
        const F2 pdf = f2_mul(f2_pack(ex2_approx(a0), ex2_approx(a1)), f2_splat(0.39894228040143268f));
        f2_unpack(f2_mul(g, f2_add(gelu_cdf2<SHORT>(v), f2_mul(v, pdf))), y[0].v[i], y[0].v[i + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float g = x[0].v[i];
        if (UOP == UN_SCALE) {
          y[0].v[i] = __fmul_rn(alpha, g);
        } else {
          const float v = x[1].v[i];
          // phi(v) = exp(-v^2 / 2) / sqrt(2 pi) = 2^(-(log2 e / 2) v^2) / sqrt(2 pi)
          const float pdf = __fmul_rn(ex2_approx(__fmul_rn(__fmul_rn(-0.72134752044448170f, v), v)),
                                      0.39894228040143268f);
          y[0].v[i] = __fmul_rn(g, __fadd_rn(gelu_cdf<SHORT>(v), __fmul_rn(v, pdf)));
        }
      }
    }
  }
};

// Copy (sum-to-shape onto the same shape).
struct CopyF {
  static constexpr bool kR1 = false, kR2 = false;
  static constexpr int kMinBlocks = kOccEwCopy;
  static constexpr int kMinBlocksWide = kOccEwCopy;
  template <int VEC>
  __device__ __forceinline__ void operator()(const Vec<VEC> (&x)[3], Vec<VEC> (&y)[2], float) const {
    y[0] = x[0];
  }
};

// ---------------------------------------------------------------- elementwise

// Slot 1 or slot 2 holds one value for every element (read once per
// thread), when the functor says so.
template <class F, class = void>
struct Uniform1 { static constexpr bool value = false; };
template <class F>
struct Uniform1<F, decltype(void(F::kUniform1))> { static constexpr bool value = F::kUniform1; };
template <class F, class = void>
struct Uniform2 { static constexpr bool value = false; };
template <class F>
struct Uniform2<F, decltype(void(F::kUniform2))> { static constexpr bool value = F::kUniform2; };

// Items each thread loads before it computes any (per pass of the elementwise
// kernels' loops): 4, or the functor's kUnroll.
template <class F, class = void>
struct ItemsPerPass { static constexpr int value = 4; };
template <class F>
struct ItemsPerPass<F, decltype(void(F::kUnroll))> { static constexpr int value = F::kUnroll; };

// One CTA = one tile of rows x column vectors.  Each thread takes items
// threadIdx.x + k * 256; items are processed in batches of U so that U
// independent loads per operand are in flight before any result is stored.
// CTAs per SM a functor's 8-wide (bfloat16) instantiation keeps.
template <class F, class = void>
struct WideBlocks { static constexpr int value = wide_occ(F::kMinBlocks); };
template <class F>
struct WideBlocks<F, decltype(void(F::kMinBlocksWide))> { static constexpr int value = F::kMinBlocksWide; };

template <class F, int VEC, int NOUT, class E = float>
__global__ void __launch_bounds__(kThreads, VEC == 8 ? WideBlocks<F>::value : F::kMinBlocks)
k_elementwise(const __grid_constant__ EwPlan p) {
  pdl_trigger();
  const E* in0 = reinterpret_cast<const E*>(p.in[0]);
  const E* in1 = reinterpret_cast<const E*>(p.in[1]);
  const E* in2 = reinterpret_cast<const E*>(p.in[2]);
  E* out0 = reinterpret_cast<E*>(p.out[0]);
  E* out1 = reinterpret_cast<E*>(p.out[1]);
  extern __shared__ int64_t s_off[];  // [tile_rows][kMaxOperands]
  const EwTile t = ew_tile(p, blockIdx.x);
  for (uint32_t i = threadIdx.x; i < t.nrows; i += blockDim.x) {
    int64_t off[kMaxOperands];
    decomp_offsets(p.rows, t.row0 + i, off);
#pragma unroll
    for (int k = 0; k < kMaxOperands; ++k) s_off[i * kMaxOperands + k] = off[k];
  }
  __syncthreads();
  pdl_wait();
  constexpr bool kUni1 = Uniform1<F>::value;
  constexpr bool kUni2 = Uniform2<F>::value;
  float uni1 = 0.f, uni2 = 0.f;
  if (kUni1) uni1 = ld1(in1, false);
  if (kUni2) uni2 = ld1(in2, false);

  constexpr int U = ItemsPerPass<F>::value;
  const F f;
  for (uint32_t it0 = 0; it0 < p.items_per_cta; it0 += U * blockDim.x) {
    Raw<E, VEC> xr[U][3];
    int64_t doff[U];
    uint32_t col[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t item = it0 + u * blockDim.x + threadIdx.x;
      const uint32_t ri = fd_div(p.tile_vcols_div, item);
      const uint32_t vc = item - ri * p.tile_vcols;
      ok[u] = ri < t.nrows && vc < t.nvcols;
      col[u] = (t.vcol0 + vc) * VEC;
      doff[u] = 0;
      if (ok[u]) {
        const int64_t* ro = s_off + ri * kMaxOperands;
        xr[u][0] = load_raw<VEC>(in0, ro[0], p.inner_stride[0], col[u], p.stream_mask & 1);
        if (F::kR1 && !kUni1)
          xr[u][1] = load_raw<VEC>(in1, ro[1], p.inner_stride[1], col[u], p.stream_mask & 2);
        if (F::kR2 && !kUni2)
          xr[u][2] = load_raw<VEC>(in2, ro[2], p.inner_stride[2], col[u], p.stream_mask & 4);
        doff[u] = ro[kSlotOut];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!ok[u]) continue;
      Vec<VEC> x[3], y[2];
      x[0] = unpack<VEC>(xr[u][0]);
      if (F::kR1 && kUni1) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[1].v[i] = uni1;
      } else if (F::kR1) {
        x[1] = unpack<VEC>(xr[u][1]);
      }
      if (F::kR2 && kUni2) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[2].v[i] = uni2;
      } else if (F::kR2) {
        x[2] = unpack<VEC>(xr[u][2]);
      }
      f(x, y, p.alpha);
      if (out0) store_cols<VEC>(out0, doff[u], p.inner_stride[kSlotOut], col[u], y[0]);
      if (NOUT > 1 && out1) store_cols<VEC>(out1, doff[u], p.inner_stride[kSlotOut], col[u], y[1]);
    }
  }
}

// Flat elementwise kernel (EwPlan with flat = 1): the same functors and loads
// as k_elementwise for problems with at most one outer dim (same-shape,
// scalar, bias-like rows), with no offset table, no barrier and no
// shared memory.  A CTA's items are consecutive in row-major order and come
// in whole batches of 1024 (U * 256 each pass of the loop), so every pass
// issues U loads per operand from every thread; each pass's u-th group of
// 256 items is 256 consecutive vectors (coalesced).
template <class F, int VEC, int NOUT, class E = float>
__global__ void __launch_bounds__(kThreads, VEC == 8 ? WideBlocks<F>::value : F::kMinBlocks)
k_flat(const __grid_constant__ EwPlan p) {
  pdl_trigger();
  const E* in0 = reinterpret_cast<const E*>(p.in[0]);
  const E* in1 = reinterpret_cast<const E*>(p.in[1]);
  const E* in2 = reinterpret_cast<const E*>(p.in[2]);
  E* out0 = reinterpret_cast<E*>(p.out[0]);
  E* out1 = reinterpret_cast<E*>(p.out[1]);
  const uint32_t first = blockIdx.x * p.items_per_cta;
  const uint32_t left = p.nitems - first;
  const uint32_t end = first + (left < p.items_per_cta ? left : p.items_per_cta);
  pdl_wait();
  constexpr bool kUni1 = Uniform1<F>::value;
  constexpr bool kUni2 = Uniform2<F>::value;
  float uni1 = 0.f, uni2 = 0.f;
  if (kUni1) uni1 = ld1(in1, false);
  if (kUni2) uni2 = ld1(in2, false);

  constexpr int U = ItemsPerPass<F>::value;
  const F f;
  for (uint32_t it0 = first; it0 < end; it0 += U * kThreads) {
    Raw<E, VEC> xr[U][3];
    int64_t doff[U];
    uint32_t col[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t item = it0 + u * kThreads + threadIdx.x;
      ok[u] = item < end;
      const uint32_t row = fd_div(p.nvcol_div, item);
      col[u] = (item - row * p.nvcol) * VEC;
      doff[u] = int64_t(row) * p.rows.stride[kSlotOut][0];
      if (ok[u]) {
        xr[u][0] = load_raw<VEC>(in0, int64_t(row) * p.rows.stride[0][0], p.inner_stride[0], col[u],
                                 p.stream_mask & 1);
        if (F::kR1 && !kUni1)
          xr[u][1] = load_raw<VEC>(in1, int64_t(row) * p.rows.stride[1][0], p.inner_stride[1],
                                   col[u], p.stream_mask & 2);
        if (F::kR2 && !kUni2)
          xr[u][2] = load_raw<VEC>(in2, int64_t(row) * p.rows.stride[2][0], p.inner_stride[2],
                                   col[u], p.stream_mask & 4);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!ok[u]) continue;
      Vec<VEC> x[3], y[2];
      x[0] = unpack<VEC>(xr[u][0]);
      if (F::kR1 && kUni1) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[1].v[i] = uni1;
      } else if (F::kR1) {
        x[1] = unpack<VEC>(xr[u][1]);
      }
      if (F::kR2 && kUni2) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[2].v[i] = uni2;
      } else if (F::kR2) {
        x[2] = unpack<VEC>(xr[u][2]);
      }
      f(x, y, p.alpha);
      if (out0) store_cols<VEC>(out0, doff[u], p.inner_stride[kSlotOut], col[u], y[0]);
      if (NOUT > 1 && out1) store_cols<VEC>(out1, doff[u], p.inner_stride[kSlotOut], col[u], y[1]);
    }
  }
}

// Launch of an elementwise plan: the flat kernel for flat plans, else the
// tiled one with its offset table in dynamic shared memory.
template <class F, int VEC, int NOUT, class E = float>
cudaError_t launch_ew_kernel(const EwPlan& p, cudaStream_t s) {
  if (p.flat) return launch_k(k_flat<F, VEC, NOUT, E>, p.n_cta, kThreads, 0, s, p);
  const size_t smem = size_t(p.tile_rows) * kMaxOperands * sizeof(int64_t);
  return launch_k(k_elementwise<F, VEC, NOUT, E>, p.n_cta, kThreads, smem, s, p);
}

// ------------------------------------------------ bfloat16 GeLU by table
//
// A bfloat16 operand takes at most 2^16 values.  On 2^-24 <= |x| < 2^8 (32
// binades of 128 values for each sign: 8192 values) GeLU on bfloat16
// storage reads its result from a table in shared memory instead of
// evaluating erfc per element: the forward's bfloat16 result, or the
// backward's derivative Phi(x) + x phi(x) in binary32, which the kernel
// multiplies by g (the product the arithmetic path rounds).  Each CTA fills
// the table with the functors themselves (the backward's with g = 1, an
// exact product), so every result is bit for bit the arithmetic path's.
// Elements outside the range (|x| < 2^-24, |x| >= 256, infinities, NaN) are
// evaluated again through the functors, in a branch taken only by warps
// that hold one.  One CTA of 1024 threads per SM, each taking an equal
// contiguous run of the items; the loads of the next pass are issued before
// the lookups of the current one.
//
// Table slot of a bfloat16 pattern b: t = (b - pattern of 2^-24) mod 2^16 is
// in [0, 4096) for 2^-24 <= x < 256 and in [32768, 36864) for their
// negatives; the slot is t & 0x8FFF, one mask.  Slots [4096, 32768) are
// never filled: a pattern outside the range reads one of them, or a filled
// slot, and is replaced.
constexpr uint32_t kGeluTabLo = (127u - 24u) << 7;  // bfloat16 pattern of 2^-24
constexpr uint32_t kGeluTabSlots = 0x9000u;
template <bool BWD>
struct GeluTab {
  static constexpr size_t kSmemBytes = size_t(kGeluTabSlots) * (BWD ? 4 : 2);
};
__device__ __forceinline__ uint32_t gelu_tab_t(uint32_t bits) { return (bits - kGeluTabLo) & 0xFFFFu; }
__device__ __forceinline__ bool gelu_tab_in(uint32_t t) { return (t & 0x7000u) == 0; }
// The k-th of the 8192 filled slots, and the value it holds the result for.
__device__ __forceinline__ uint32_t gelu_nth_slot(uint32_t k) {
  return k < 4096u ? k : k - 4096u + 0x8000u;
}
__device__ __forceinline__ float gelu_slot_value(uint32_t slot) {
  return __uint_as_float(((slot + kGeluTabLo) & 0xFFFFu) << 16);
}

// Elements outside the table, one at a time through the functors.
__device__ __forceinline__ uint32_t gelu_fwd_bf16_slow(uint32_t bits) {
  Vec<1> x[3], y[2];
  x[0].v[0] = __uint_as_float(bits << 16);
  UnaryF<UN_GELU, true>{}(x, y, 0.f);
  return __bfloat16_as_ushort(__float2bfloat16_rn(y[0].v[0]));
}
__device__ __forceinline__ float gelu_bwd_bf16_slow(float g, uint32_t bits) {
  Vec<1> x[3], y[2];
  x[0].v[0] = g;
  x[1].v[0] = __uint_as_float(bits << 16);
  UnaryBwdF<UN_GELU, true>{}(x, y, 0.f);
  return y[0].v[0];
}

template <bool BWD>
__device__ __forceinline__ void gelu_fill(uint32_t* tab) {
  for (uint32_t k = threadIdx.x; k < 4096u; k += kGeluTabThreads) {
    const uint32_t s = gelu_nth_slot(2 * k);  // slots s, s + 1
    Vec<2> x[3], y[2];
    if constexpr (BWD) {
      x[0].v[0] = x[0].v[1] = 1.f;
      x[1].v[0] = gelu_slot_value(s);
      x[1].v[1] = gelu_slot_value(s + 1);
      UnaryBwdF<UN_GELU, true>{}(x, y, 0.f);
      *reinterpret_cast<uint2*>(tab + s) = make_uint2(__float_as_uint(y[0].v[0]), __float_as_uint(y[0].v[1]));
    } else {
      x[0].v[0] = gelu_slot_value(s);
      x[0].v[1] = gelu_slot_value(s + 1);
      UnaryF<UN_GELU, true>{}(x, y, 0.f);
      tab[s / 2] = pack_bf16x2(y[0].v[0], y[0].v[1]);
    }
  }
}

template <int VEC>
__device__ __forceinline__ uint32_t raw_bits(const Raw<__nv_bfloat16, VEC>& r, int i) {
  return (i & 1) ? r.w[i / 2] >> 16 : r.w[i / 2] & 0xFFFFu;
}

// The results of one item: forward bfloat16 patterns, backward values.
// `lanes`: the lanes of the warp that call it for this item (the vote names
// exactly them).
template <int VEC>
__device__ __forceinline__ void gelu_item_fwd(const uint32_t* tab, unsigned lanes,
                                              const Raw<__nv_bfloat16, VEC>& xr,
                                              uint32_t (&w)[(VEC + 1) / 2]) {
  const unsigned short* th = reinterpret_cast<const unsigned short*>(tab);
  uint32_t bad = 0;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const uint32_t t = gelu_tab_t(raw_bits<VEC>(xr, i));
    bad |= t & 0x7000u;
    const uint32_t r = th[t & 0x8FFFu];
    if (i & 1) w[i / 2] |= r << 16;
    else w[i / 2] = r;
  }
  if (__any_sync(lanes, bad != 0)) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const uint32_t bits = raw_bits<VEC>(xr, i);
      if (!gelu_tab_in(gelu_tab_t(bits))) {
        const uint32_t r = gelu_fwd_bf16_slow(bits);
        w[i / 2] = (i & 1) ? (w[i / 2] & 0xFFFFu) | (r << 16) : (w[i / 2] & 0xFFFF0000u) | r;
      }
    }
  }
}
template <int VEC>
__device__ __forceinline__ void gelu_item_bwd(const uint32_t* gsm, unsigned lanes,
                                              const Raw<__nv_bfloat16, VEC>& xr,
                                              const Raw<__nv_bfloat16, VEC>& gr, Vec<VEC>& y) {
  const float* tf = reinterpret_cast<const float*>(gsm);
  uint32_t bad = 0;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const uint32_t t = gelu_tab_t(raw_bits<VEC>(xr, i));
    bad |= t & 0x7000u;
    y.v[i] = __fmul_rn(__uint_as_float(raw_bits<VEC>(gr, i) << 16), tf[t & 0x8FFFu]);
  }
  if (__any_sync(lanes, bad != 0)) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const uint32_t bits = raw_bits<VEC>(xr, i);
      if (!gelu_tab_in(gelu_tab_t(bits)))
        y.v[i] = gelu_bwd_bf16_slow(__uint_as_float(raw_bits<VEC>(gr, i) << 16), bits);
    }
  }
}

// Store VEC bfloat16 patterns, two per word, as store_cols stores values.
template <int VEC>
__device__ __forceinline__ void store_raw_bf16(__nv_bfloat16* base, int64_t row_off, int64_t inner,
                                               uint32_t c, const uint32_t (&w)[(VEC + 1) / 2]) {
  unsigned short* b = reinterpret_cast<unsigned short*>(base) + row_off;
  if (inner == 1) {
    if constexpr (VEC == 8) {
      *reinterpret_cast<uint4*>(b + c) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (VEC == 4) {
      *reinterpret_cast<uint2*>(b + c) = make_uint2(w[0], w[1]);
    } else {
      static_assert(VEC == 1, "vector width");
      b[c] = static_cast<unsigned short>(w[0]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i)
      b[int64_t(c + i) * inner] = static_cast<unsigned short>((i & 1) ? w[i / 2] >> 16 : w[i / 2]);
  }
}

// in0: x (forward) or g (backward), in1: x (backward); a flat plan; dynamic
// shared memory GeluTab<BWD>::kSmemBytes.  U items per pass.
template <bool BWD, int VEC>
__global__ void __launch_bounds__(kGeluTabThreads, 1)
k_gelu_bf16(const __grid_constant__ EwPlan p) {
  using E = __nv_bfloat16;
  extern __shared__ __align__(16) uint32_t gsm[];
  constexpr int U = BWD ? kGeluTabUnrollBwd : kGeluTabUnrollFwd;
  constexpr uint32_t kStep = U * kGeluTabThreads;
  pdl_trigger();
  const uint32_t first = uint32_t(uint64_t(p.nitems) * blockIdx.x / gridDim.x);
  const uint32_t end = uint32_t(uint64_t(p.nitems) * (blockIdx.x + 1) / gridDim.x);
  const int xs = BWD ? 1 : 0;
  const E* xin = reinterpret_cast<const E*>(p.in[xs]);
  const E* gin = reinterpret_cast<const E*>(p.in[0]);
  E* out = reinterpret_cast<E*>(p.out[0]);
  struct Pass {
    Raw<E, VEC> xr[U], gr[U];
  };
  auto load = [&](uint32_t it0, Pass& q) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t item = it0 + u * kGeluTabThreads + threadIdx.x;
      if (item < end) {
        const uint32_t row = fd_div(p.nvcol_div, item);
        const uint32_t col = (item - row * p.nvcol) * VEC;
        q.xr[u] = load_raw<VEC>(xin, int64_t(row) * p.rows.stride[xs][0], p.inner_stride[xs], col,
                                p.stream_mask & (1u << xs));
        if (BWD)
          q.gr[u] = load_raw<VEC>(gin, int64_t(row) * p.rows.stride[0][0], p.inner_stride[0], col,
                                  p.stream_mask & 1);
      }
    }
  };
  pdl_wait();
  // The first pass's loads are in flight while the table is filled.
  Pass cur, nxt;
  load(first, cur);
  gelu_fill<BWD>(gsm);
  __syncthreads();
  for (uint32_t it0 = first; it0 < end; it0 += kStep) {
    if (it0 + kStep < end) load(it0 + kStep, nxt);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t item = it0 + u * kGeluTabThreads + threadIdx.x;
      const unsigned lanes = __ballot_sync(0xffffffffu, item < end);
      if (item >= end) continue;
      const uint32_t row = fd_div(p.nvcol_div, item);
      const uint32_t col = (item - row * p.nvcol) * VEC;
      const int64_t doff = int64_t(row) * p.rows.stride[kSlotOut][0];
      if constexpr (BWD) {
        Vec<VEC> y;
        gelu_item_bwd<VEC>(gsm, lanes, cur.xr[u], cur.gr[u], y);
        store_cols<VEC>(out, doff, p.inner_stride[kSlotOut], col, y);
      } else {
        uint32_t w[(VEC + 1) / 2];
        gelu_item_fwd<VEC>(gsm, lanes, cur.xr[u], w);
        store_raw_bf16<VEC>(out, doff, p.inner_stride[kSlotOut], col, w);
      }
    }
    cur = nxt;
  }
}

// Forward with a transposed input (TrPlan): x has unit stride along p, the
// output along q.  A CTA covers kTrP p x kTrTile q; warp w its p rows
// [16w, 16w + 16), lane (pc = lane & 3, qq = lane >> 2) a 4 x 4 block at
// p = 4 pc, q = 4 qq.  The block is read as four 16-byte loads along p (one
// per q; a warp's load covers 64 contiguous bytes in each of 8 rows),
// transposed in registers and written as four 16-byte stores along q (a
// warp's store covers 128 contiguous bytes in each of 4 rows): no shared
// memory and no barrier.  Blocks cut by the edge of p or q, or views
// without 16-byte alignment, use scalar accesses with the same mapping.
template <int OP>
__global__ void __launch_bounds__(kThreads, kOccTr)
k_transpose(const __grid_constant__ TrPlan p) {
  pdl_trigger();
  const uint32_t t1 = fd_div(p.n_qt_div, blockIdx.x);
  const uint32_t qt = blockIdx.x - t1 * p.n_qt;
  const uint32_t bidx = fd_div(p.n_pt_div, t1);
  const uint32_t pt = t1 - bidx * p.n_pt;
  int64_t base[kMaxOperands];
  decomp_offsets(p.batch, bidx, base);
  const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t ps = pt * kTrP + 16 * w + 4 * (lane & 3);  // this thread's first p
  const uint32_t qs = qt * kTrTile + 4 * (lane >> 2);       // and first q
  if (ps >= p.np || qs >= p.nq) return;
  const float* __restrict__ x = p.x + base[0];
  const float* __restrict__ y = p.y + base[1];
  float* __restrict__ out = p.out + base[kSlotOut];
  const bool fast = p.vec_ok && ps + 4 <= p.np && qs + 4 <= p.nq;
  const uint32_t np4 = min(4u, p.np - ps), nq4 = min(4u, p.nq - qs);
  pdl_wait();

  float v[4][4];  // [q][p]
  if (fast) {
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k) {
      const float4 t = __ldcs(reinterpret_cast<const float4*>(x + ps + int64_t(qs + k) * p.xs_q));
      v[k][0] = t.x; v[k][1] = t.y; v[k][2] = t.z; v[k][3] = t.w;
    }
  } else {
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k)
#pragma unroll
      for (uint32_t c = 0; c < 4; ++c)
        v[k][c] = (k < nq4 && c < np4) ? __ldcs(x + ps + c + int64_t(qs + k) * p.xs_q) : 0.f;
  }
  // y at (p, q); a y broadcast along q or p is loaded once per row/column.
  float yv[4][4];  // [p][q]
  if (p.ys_q == 0) {
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c) {
      const float t = c < np4 ? __ldg(y + int64_t(ps + c) * p.ys_p) : 0.f;
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k) yv[c][k] = t;
    }
  } else if (p.ys_p == 0) {
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k) {
      const float t = k < nq4 ? __ldg(y + int64_t(qs + k) * p.ys_q) : 0.f;
#pragma unroll
      for (uint32_t c = 0; c < 4; ++c) yv[c][k] = t;
    }
  } else {
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c)
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k)
        yv[c][k] = (c < np4 && k < nq4)
                       ? __ldg(y + int64_t(ps + c) * p.ys_p + int64_t(qs + k) * p.ys_q) : 0.f;
  }
  float r[4][4];  // [p][q]
#pragma unroll
  for (uint32_t c = 0; c < 4; ++c)
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k)
      r[c][k] = p.x_is_a ? fwd_op<OP>(v[k][c], yv[c][k]) : fwd_op<OP>(yv[c][k], v[k][c]);
  if (fast) {
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c)
      *reinterpret_cast<float4*>(out + int64_t(ps + c) * p.os_p + qs) =
          make_float4(r[c][0], r[c][1], r[c][2], r[c][3]);
  } else {
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c)
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k)
        if (c < np4 && k < nq4) out[int64_t(ps + c) * p.os_p + qs + k] = r[c][k];
  }
}

// Split forward (SabFPlan): CTA = (tile of a's rows, chunk of betas).
// Thread (tx, ty) holds a's float4 at column tx for rows ty, ty + lanes, ...
// and writes them against each beta's b row: one load of b per beta, one
// operation and one 16-byte store per four outputs.
template <int OP, int RPT>
__global__ void __launch_bounds__(kThreads, kOccSabf)
k_sabf(const __grid_constant__ SabFPlan p) {
  pdl_trigger();
  const uint32_t tile = fd_div(p.n_bc_div, blockIdx.x);
  const uint32_t bc = blockIdx.x - tile * p.n_bc;
  const uint32_t nvc = p.nvc;
  const uint32_t nvc_shift = __ffs(nvc) - 1;
  const uint32_t lanes = kThreads >> nvc_shift;
  const uint32_t tx = threadIdx.x & (nvc - 1);
  const uint32_t ty = threadIdx.x >> nvc_shift;
  int64_t ob[kMaxOperands];
  decomp_offsets(p.a_outer, tile, ob);
  int64_t aoff[RPT], ooff[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
    int64_t ri[kMaxOperands];
    decomp_offsets(p.a_inner, ty + j * lanes, ri);
    aoff[j] = ob[1] + ri[1] + tx * 4;
    ooff[j] = ob[0] + ri[0] + tx * 4;
  }
  pdl_wait();
  float4 areg[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) areg[j] = __ldg(reinterpret_cast<const float4*>(p.a + aoff[j]));
  const uint32_t b0 = bc * p.beta_chunk;
  const uint32_t b1 = min(p.n_beta, b0 + p.beta_chunk);
  for (uint32_t beta = b0; beta < b1; ++beta) {
    int64_t bo[kMaxOperands];
    decomp_offsets(p.beta, beta, bo);
    const float4 b4 = __ldg(reinterpret_cast<const float4*>(p.b + bo[2] + tx * 4));
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const float4 r = make_float4(fwd_op<OP>(areg[j].x, b4.x), fwd_op<OP>(areg[j].y, b4.y),
                                   fwd_op<OP>(areg[j].z, b4.z), fwd_op<OP>(areg[j].w, b4.w));
      // Evict-first stores: the 3 GB written here is never read back by
      // this kernel (c5b's forward 466.9 -> 440.1 us; the same hint on the
      // flat and reduction kernels measured no faster).
      __stcs(reinterpret_cast<float4*>(p.out + ooff[j] + bo[0]), r);
    }
  }
}

// ---------------------------------------------------------------- reduction

// Term of the reduced gradient X (WHICH: 0 = a, 1 = b; 2 = sum-to-shape
// identity) and, when the other gradient is written densely in the same pass,
// the other term.
template <int OP, int WHICH, bool SHORT = false>
struct RedTerms {
  // div with grad_b reduced: b is constant along the reduction (it is the
  // broadcast operand), so sum(-g*a/b^2) = -(1/b^2) * sum(g*a): the kernel adds
  // g*a and applies post(b) once per output.
  static constexpr bool kPost = OP == OP_DIV && WHICH == 1;
  // Inputs read per element by X's term, and by the dense gradient's term
  // (only when a dense gradient is written in the same pass).
  static constexpr bool kXa = Needs<OP, WHICH>::a;
  static constexpr bool kXb = Needs<OP, WHICH>::b && !kPost;
  static constexpr bool kDa = WHICH < 2 && Needs<OP, 1 - WHICH>::a;
  static constexpr bool kDb = WHICH < 2 && Needs<OP, 1 - WHICH>::b;
  // Summed terms need not be single IEEE operations (the sum is within
  // tolerance, not bit-exact): div's g/b is taken as g * (1/b).
  // X's term is g * m(a, b); the kernel adds the product through an FMA.
  __device__ __forceinline__ static float m(float a, float b) {
    if (WHICH == 0) {
      if (OP == OP_MUL) return b;
      if (OP == OP_DIV) return __frcp_rn(b);
      return 1.0f;
    }
    if (WHICH == 1) {
      if (OP == OP_SUB) return -1.0f;
      if (OP == OP_MUL || OP == OP_DIV) return a;
      return 1.0f;
    }
    return 1.0f;
  }
  __device__ __forceinline__ static float post(float b) {
    const float r = __frcp_rn(b);
    return -__fmul_rn(r, r);
  }
  // Dense gradient terms stay exact single operations (bit-identical).
  template <int VEC>
  __device__ __forceinline__ static void d(const Vec<VEC>& g, const Vec<VEC>& a, const Vec<VEC>& b,
                                           Vec<VEC>& out) {
    if (WHICH == 0) term_b_vec<OP, SHORT>(g, a, b, out);
    else term_a_vec<OP, SHORT>(g, a, b, out);
  }
  // The same rule on the host: which pointers the kernel dereferences.
  static bool reads_a(bool has_d) { return kXa || (has_d && kDa); }
  static bool reads_b(bool has_d) { return kXb || (has_d && kDb) || kPost; }
};

// Reduction pass.  CTA = (kept index, row block, column block).  Rows of
// the block come from a shared-memory offset table (reduced outer dims,
// refilled every kMaxTileRows rows), the kept index adds a CTA-wide base
// offset.  INNER_KEPT: thread (tx, ty) owns column vector tx of the block and
// adds rows ty, ty + ty_n, ...; then a fixed tree over ty.  Otherwise every
// thread adds its rows and columns into one value and the CTA reduces them
// with a fixed tree.  Per-thread sums are Kahan-compensated, so the error
// bound does not grow with the number of rows a thread adds.
//
// CL (cluster plans): the CTAs of one output tile form a cluster; each keeps
// its tree result in shared memory, and after a cluster barrier the rank-0
// CTA adds the cluster's results in rank order and writes X.  A second
// barrier keeps every CTA resident until the leader has read it.  CL kernels
// keep more items in flight per thread (red_cl_unroll).
template <int OP, int WHICH, int VEC, bool INNER_KEPT, bool CL = false, class E = float>
__global__ void __launch_bounds__(kThreads,
                                  CL ? red_cl_occ(OP, INNER_KEPT)
                                     : (VEC == 8 ? red_wide_occ(OP, INNER_KEPT)
                                                 : ((OP == OP_MUL || OP == OP_DIV) ? kOccRedMulDiv
                                                                                  : kOccRedAddSub)))
k_reduce(const __grid_constant__ RedPlan p) {
  pdl_trigger();
  // Operands and gradients in storage type E; partial slots are binary32.
  const E* gE = reinterpret_cast<const E*>(p.g);
  const E* aE = reinterpret_cast<const E*>(p.a);
  const E* bE = reinterpret_cast<const E*>(p.b);
  E* xE = reinterpret_cast<E*>(p.x_final);
  E* dE = reinterpret_cast<E*>(p.d_out);
  // bfloat16 operands divide by the forms for short operands (term_a_vec,
  // term_b_vec).
  using T = RedTerms<OP, WHICH, sizeof(E) == 2>;
  extern __shared__ int64_t s_dyn[];
  const uint32_t table_rows = p.rows_per_blk < kMaxTileRows ? p.rows_per_blk : kMaxTileRows;
  int64_t* s_off = s_dyn;  // [table_rows][kMaxOperands]
  float* s_red = reinterpret_cast<float*>(s_dyn + kMaxOperands * table_rows);
  // Staging ring (p.stages > 0): [stages][stage_ns][4][kThreads] 16-byte
  // slots.  It shares its memory with the tree (s_red), which is written
  // only after every thread has finished its loads and passed a barrier.
  uint4* s_stage = reinterpret_cast<uint4*>(s_red);

  const RedCta cta = red_cta(p, blockIdx.x);
  int64_t base[kMaxOperands];
  decomp_offsets(p.kept, cta.kidx, base);
  const uint32_t row0 = cta.rblk * p.rows_per_blk;
  const uint32_t rleft = p.n_red - row0;
  const uint32_t nrows = rleft < p.rows_per_blk ? rleft : p.rows_per_blk;

  const uint32_t tx = threadIdx.x % p.tx;
  const uint32_t ty = threadIdx.x / p.tx;
  const bool has_d = p.d_out != nullptr;
  const bool read_a = T::kXa || (has_d && T::kDa);
  const bool read_b = T::kXb || (has_d && T::kDb);
  const uint32_t vcol_begin = cta.cblk * p.vcols_per_blk;
  const uint32_t vcol_end_raw = vcol_begin + p.vcols_per_blk;
  const uint32_t vcol_end = vcol_end_raw < p.nvcol ? vcol_end_raw : p.nvcol;

  Kahan acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i].init();
  // Column vectors this thread owns in the block (one when the inner dim is
  // kept: vcols_per_blk == tx).
  const uint32_t ncs = vcol_end > vcol_begin + tx ? (vcol_end - vcol_begin - tx + p.tx - 1) / p.tx : 0;
  // The input of the gradient being reduced (a for grad_a, b for grad_b) is
  // broadcast along every reduced dim, so its value depends only on the kept
  // index and, when the inner dim is kept, the column: loaded once, after the
  // first chunk's offset table (parameters only) is built and pdl_wait().
  Vec<VEC> own;
#pragma unroll
  for (int i = 0; i < VEC; ++i) own.v[i] = 0.f;
  // div with grad_b reduced: the dense gradient is g / b with b = own, and
  // own serves nothing else (grad_b's own factor is applied once, by post).
  // For bfloat16 storage, when every lane of own is a power of two, own is
  // replaced by 1/b and the dense gradient is g * own, bit for bit
  // (pow2_reciprocal): c4's backward division in bf16 103 -> 96 us.  Float
  // storage keeps the IEEE division there: it is not what bounds that
  // kernel, and the flag's registers made it spill.
  constexpr bool kP2 = OP == OP_DIV && WHICH == 1 && sizeof(E) == 2;
  bool own_p2 = false;

  for (uint32_t ch0 = 0; ch0 < nrows; ch0 += kMaxTileRows) {
    const uint32_t cleft = nrows - ch0;
    const uint32_t nch = cleft < kMaxTileRows ? cleft : kMaxTileRows;
    if (ch0 > 0) __syncthreads();
    for (uint32_t i = threadIdx.x; i < nch; i += blockDim.x) {
      int64_t off[kMaxOperands];
      decomp_offsets(p.red, row0 + ch0 + i, off);
#pragma unroll
      for (int k = 0; k < kMaxOperands; ++k) s_off[i * kMaxOperands + k] = off[k] + base[k];
    }
    __syncthreads();
    if (ch0 == 0) {
      pdl_wait();
      if (WHICH < 2 && ncs > 0) {
        const int slot = WHICH == 0 ? 1 : 2;
        const bool needed =
            WHICH == 0 ? ((T::kXa || T::kDa) && read_a) : ((T::kXb || T::kDb) && read_b);
        if (needed)
          own = load_cols<VEC>(WHICH == 0 ? aE : bE, base[slot], p.inner_stride[slot],
                               (vcol_begin + tx) * VEC, false);
        if (kP2 && needed) {
          Vec<VEC> r;
          bool p2 = true;
#pragma unroll
          for (int i = 0; i < VEC; ++i) p2 = pow2_reciprocal(own.v[i], &r.v[i]) && p2;
          if (p2) {
            own = r;
            own_p2 = true;
          }
        }
      }
    }

    // This thread's items are (row, column vector) pairs: rows ty, ty + ty_n,
    // ... of the chunk, columns vcol_begin + tx, + tx_n, ... of the block,
    // walked columns-fastest and loaded U at a time so that U independent
    // loads per operand are in flight whichever of the two is longer.
    const uint32_t nrs = nch > ty ? (nch - ty + p.ty - 1) / p.ty : 0;
    const uint32_t items = ncs * nrs;
    uint32_t rm = 0, cm = 0;
    constexpr int U = CL ? red_cl_unroll(OP) : 4;
    // bfloat16 with the inner dim reduced: a vector's 8 products are added
    // by a 3-level tree before the per-thread Kahan sum (fewer instructions
    // for the 2-byte stream; the products' roundings and the tree add at
    // most 4u of each term's size, far inside the tolerance).
    constexpr bool kPairwise = !INNER_KEPT && sizeof(E) == 2;
    // Inputs streamed per item besides g: a (when X is grad_b or the dense
    // gradient needs it) or b (likewise).
    constexpr bool kSA = (T::kXa || T::kDa) && WHICH != 0;
    constexpr bool kSB = (T::kXb || T::kDb) && WHICH != 1;
    const bool sa = kSA && read_a, sb = kSB && read_b;
    // One item: row ri of the chunk, columns cc .. cc + VEC - 1.
    auto proc = [&](const Raw<E, VEC>& gr, const Raw<E, VEC>& ar, const Raw<E, VEC>& br, uint32_t ri,
                    uint32_t cc) {
      const Vec<VEC> gv = unpack<VEC>(gr);
      Vec<VEC> av, bv;
      if (kSA && sa) av = unpack<VEC>(ar);
      if (kSB && sb) bv = unpack<VEC>(br);
      Vec<VEC> aw, bw;
      float pr[VEC];
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        const float aa = ((T::kXa || T::kDa) && read_a) ? (WHICH == 0 ? own.v[i] : av.v[i]) : 0.f;
        const float bb = ((T::kXb || T::kDb) && read_b) ? (WHICH == 1 ? own.v[i] : bv.v[i]) : 0.f;
        aw.v[i] = aa;
        bw.v[i] = bb;
        if (INNER_KEPT) acc[i].add_prod(gv.v[i], T::m(aa, bb));
        else if (kPairwise) pr[i] = __fmul_rn(gv.v[i], T::m(aa, bb));
        else acc[0].add_prod(gv.v[i], T::m(aa, bb));
      }
      if (kPairwise) {
        // The vector's products by a fixed pairwise tree, then one
        // compensated addition.
#pragma unroll
        for (int w = 1; w < VEC; w *= 2)
#pragma unroll
          for (int i = 0; i + w < VEC; i += 2 * w) pr[i] = __fadd_rn(pr[i], pr[i + w]);
        acc[0].add(pr[0]);
      }
      if (has_d) {
        Vec<VEC> dv;
        if (kP2 && own_p2) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) dv.v[i] = __fmul_rn(gv.v[i], own.v[i]);
        } else {
          T::d(gv, aw, bw, dv);
        }
        store_cols<VEC>(dE, s_off[ri * kMaxOperands + kSlotOut], p.inner_stride[kSlotOut], cc, dv);
      }
    };
    if constexpr (VEC * sizeof(E) == 16) {
      if (p.stages >= 2 && 1u + ((sa || sb) ? 1u : 0u) <= p.stage_ns) {
        // Staged: each thread copies the 16-byte vectors of its items into
        // its own slots of a ring of p.stages batches in shared memory
        // (cp.async) and reads them back once its copies of that batch have
        // landed, so p.stages - 1 further batches stay in flight while one
        // is summed, without holding registers.  Same items, same order,
        // same arithmetic as the loop below.
        const uint32_t S = p.stages, NSL = p.stage_ns;
        auto slot = [&](uint32_t st, uint32_t k, int u) {
          return s_stage + ((st * NSL + k) * U + u) * kThreads + threadIdx.x;
        };
        uint32_t irm = 0, icm = 0, im = 0;
        auto issue = [&](uint32_t st) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (im < items) {
              const uint32_t ri = ty + irm * p.ty;
              const uint32_t cc = (vcol_begin + tx + icm * p.tx) * VEC;
              const int64_t* ro = s_off + ri * kMaxOperands;
              cp_async16(slot(st, 0, u), gE + ro[0] + cc);
              if (kSA && sa) cp_async16(slot(st, 1, u), aE + ro[1] + cc);
              if (kSB && sb) cp_async16(slot(st, 1, u), bE + ro[2] + cc);
              if (++icm == ncs) { icm = 0; ++irm; }
              ++im;
            }
          }
          cp_async_commit();
        };
        for (uint32_t st = 0; st + 1 < S; ++st) issue(st);
        uint32_t st = 0;
        for (uint32_t m0 = 0; m0 < items; m0 += U) {
          issue(st == 0 ? S - 1 : st - 1);  // the slot the previous batch used
          if (S >= 3) cp_async_wait<2>();
          else cp_async_wait<1>();
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (m0 + u >= items) continue;
            const uint32_t ri = ty + rm * p.ty;
            const uint32_t cc = (vcol_begin + tx + cm * p.tx) * VEC;
            if (++cm == ncs) { cm = 0; ++rm; }
            Raw<E, VEC> gr = raw_from_u4<E, VEC>(*slot(st, 0, u)), ar, br;
            if (kSA && sa) ar = raw_from_u4<E, VEC>(*slot(st, 1, u));
            if (kSB && sb) br = raw_from_u4<E, VEC>(*slot(st, 1, u));
            proc(gr, ar, br, ri, cc);
          }
          st = st + 1 == S ? 0 : st + 1;
        }
        cp_async_wait<0>();
        continue;  // next chunk of rows
      }
    }
    for (uint32_t m0 = 0; m0 < items; m0 += U) {
      Raw<E, VEC> gr[U], ar[U], br[U];
      uint32_t ri[U], cc[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ok[u] = m0 + u < items;
        ri[u] = ty + rm * p.ty;
        cc[u] = (vcol_begin + tx + cm * p.tx) * VEC;
        if (ok[u]) {
          const int64_t* ro = s_off + ri[u] * kMaxOperands;
          gr[u] = load_raw<VEC>(gE, ro[0], p.inner_stride[0], cc[u], p.stream_mask & 1);
          if (kSA && sa) ar[u] = load_raw<VEC>(aE, ro[1], p.inner_stride[1], cc[u], p.stream_mask & 2);
          if (kSB && sb) br[u] = load_raw<VEC>(bE, ro[2], p.inner_stride[2], cc[u], p.stream_mask & 4);
          if (++cm == ncs) { cm = 0; ++rm; }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) proc(gr[u], ar[u], br[u], ri[u], cc[u]);
    }
  }

  if (INNER_KEPT) {
    // Fixed tree over the ty row lanes of each column vector (ty = 256/tx is
    // a power of two).
    const uint32_t lanes = p.tx * VEC;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < VEC; ++i) s_red[ty * lanes + tx * VEC + i] = acc[i].s;
    for (uint32_t h = p.ty >> 1; h > 0; h >>= 1) {
      __syncthreads();
      if (ty < h) {
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          s_red[ty * lanes + tx * VEC + i] =
              __fadd_rn(s_red[ty * lanes + tx * VEC + i], s_red[(ty + h) * lanes + tx * VEC + i]);
      }
    }
    __syncthreads();
    if (CL) {
      // s_red[0, lanes) holds this CTA's column sums; the leader adds the
      // cluster's in rank order.
      cluster_sync();
      if (cluster_rank() == 0) {
        for (uint32_t v = threadIdx.x; v < lanes; v += blockDim.x) {
          const uint32_t vcv = vcol_begin + v / VEC;
          const uint32_t col = vcv * VEC + v % VEC;
          if (vcv >= vcol_end || col >= p.ncol) continue;
          float r = ld_cluster(s_red + v, 0);
          for (uint32_t k = 1; k < p.cluster; ++k) r = __fadd_rn(r, ld_cluster(s_red + v, k));
          if (T::kPost) r = __fmul_rn(r, T::post(ld1(bE + base[2] + int64_t(col) * p.inner_stride[2], false)));
          st1(xE + uint64_t(cta.kidx) * p.ncol + col, __fmul_rn(r, p.scale));
        }
      }
      cluster_sync();
      return;
    }
    const uint32_t vc = vcol_begin + tx;
    if (ty == 0 && vc < vcol_end) {
      Vec<VEC> r;
      const uint64_t j = uint64_t(cta.kidx) * p.ncol + uint64_t(vc) * VEC;
#pragma unroll
      for (int i = 0; i < VEC; ++i) r.v[i] = s_red[tx * VEC + i];
      Vec<VEC> f;  // div's -1/b^2 per output
      if (T::kPost) {
        const Vec<VEC> bv = load_cols<VEC>(bE, base[2], p.inner_stride[2], vc * VEC, false);
#pragma unroll
        for (int i = 0; i < VEC; ++i) f.v[i] = T::post(bv.v[i]);
      }
      if (p.nslots == 1) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          if (T::kPost) r.v[i] = __fmul_rn(r.v[i], f.v[i]);
          r.v[i] = __fmul_rn(r.v[i], p.scale);
        }
        store_cols<VEC>(xE + j, 0, 1, 0, r);
      } else {
        // Partials stay unscaled: the second pass multiplies each total by
        // its factor, stored after the slots by the slot-0 CTAs.
        store_cols<VEC>(p.partial + uint64_t(cta.rblk) * p.nout + j, 0, 1, 0, r);
        if (T::kPost && cta.rblk == 0)
          store_cols<VEC>(p.partial + uint64_t(p.nslots) * p.nout + j, 0, 1, 0, f);
      }
    }
  } else {
    // Whole-CTA fixed tree: one value per kept index.
    __syncthreads();
    s_red[threadIdx.x] = acc[0].s;
    for (uint32_t h = blockDim.x >> 1; h > 0; h >>= 1) {
      __syncthreads();
      if (threadIdx.x < h) s_red[threadIdx.x] = __fadd_rn(s_red[threadIdx.x], s_red[threadIdx.x + h]);
    }
    if (CL) {
      cluster_sync();
      if (cluster_rank() == 0 && threadIdx.x == 0) {
        float r = ld_cluster(s_red, 0);
        for (uint32_t k = 1; k < p.cluster; ++k) r = __fadd_rn(r, ld_cluster(s_red, k));
        if (T::kPost) r = __fmul_rn(r, T::post(ld1(bE + base[2], false)));
        st1(xE + cta.kidx, __fmul_rn(r, p.scale));
      }
      cluster_sync();
      return;
    }
    if (threadIdx.x == 0) {
      float r = s_red[0];
      const float f = T::kPost ? T::post(ld1(bE + base[2], false)) : 1.0f;
      if (p.nslots == 1) {
        if (T::kPost) r = __fmul_rn(r, f);
        st1(xE + cta.kidx, __fmul_rn(r, p.scale));
      } else {
        // Unscaled partial; slot 0 also stores the factor for the second pass.
        const uint64_t slot = uint64_t(cta.rblk) * p.n_cblk + cta.cblk;
        p.partial[slot * p.nout + cta.kidx] = r;
        if (T::kPost && slot == 0) p.partial[uint64_t(p.nslots) * p.nout + cta.kidx] = f;
      }
    }
  }
}

// Second pass: for each output j, add its nslots partials in slot order (and
// multiply the total by its factor when p.post is set).
// Thread (jx lane, sy lane) adds slots sy, sy + sy_n, ... (Kahan), then a
// fixed tree over the sy lanes.  V = 4: each thread takes 4 consecutive
// outputs with 16-byte loads of the partials (more bytes in flight per
// thread; the launcher takes it when the outputs and slots are aligned).
template <class E = float, int V = 1>
static __global__ void __launch_bounds__(kThreads)
k_combine(const __grid_constant__ CombinePlan p) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_red[kThreads * V];
  const uint32_t jl = threadIdx.x % p.jx;
  const uint32_t sl = threadIdx.x / p.jx;
  const uint64_t j = (uint64_t(blockIdx.x) * p.jx + jl) * V;
  Kahan acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i].init();
  if (j < p.nout && sl < p.sy) {
    // Up to eight partials (vectors) are loaded before any is added, so
    // their loads overlap (a ragged last batch is predicated, not walked one
    // by one).
    const float* src = p.partial + uint64_t(sl) * p.nout + j;
    const uint64_t step = uint64_t(p.sy) * p.nout;
    for (uint32_t s = sl; s < p.nslots; s += 8 * p.sy, src += 8 * step) {
      Vec<V> v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool in = s + u * p.sy < p.nslots;
        if constexpr (V == 4) {
          const float4 q = in ? __ldg(reinterpret_cast<const float4*>(src + u * step))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
          v[u].v[0] = q.x; v[u].v[1] = q.y; v[u].v[2] = q.z; v[u].v[3] = q.w;
        } else {
          v[u].v[0] = in ? __ldg(src + u * step) : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (s + u * p.sy < p.nslots) {
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i].add(v[u].v[i]);
        }
    }
  }
  const uint32_t syn = blockDim.x / p.jx;  // power of two
#pragma unroll
  for (int i = 0; i < V; ++i) s_red[(sl * p.jx + jl) * V + i] = (sl < p.sy) ? acc[i].s : 0.f;
  for (uint32_t h = syn >> 1; h > 0; h >>= 1) {
    __syncthreads();
    if (sl < h) {
#pragma unroll
      for (int i = 0; i < V; ++i)
        s_red[(sl * p.jx + jl) * V + i] =
            __fadd_rn(s_red[(sl * p.jx + jl) * V + i], s_red[((sl + h) * p.jx + jl) * V + i]);
    }
  }
  __syncthreads();
  if (sl == 0 && j < p.nout) {
    E* out = reinterpret_cast<E*>(p.out);
    E* out2 = reinterpret_cast<E*>(p.out2);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const uint64_t jj = j + i;
      if (jj >= p.nout) break;
      float v = s_red[jl * V + i];
      if (p.post) v = __fmul_rn(v, __ldg(p.partial + uint64_t(p.nslots) * p.nout + jj));
      v = __fmul_rn(v, p.scale);
      st1(jj < p.split ? out + jj : out2 + (jj - p.split), v);
    }
  }
}

}  // namespace zr
