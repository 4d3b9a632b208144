// zr_launch_bf16.cu — bfloat16-storage instantiations of the elementwise,
// reduction and combine kernels (binary32 arithmetic, one rounding to bf16
// per stored element; partial sums stay binary32).  The launchers of the
// float paths hand plans with es == 2 to these.
#include <cuda_bf16.h>

#include "zr_launch.h"
#include "zr_kernels.cuh"

namespace zr {

namespace {

using bf16 = __nv_bfloat16;

template <class F, int NOUT>
cudaError_t launch_ew_bf16(const EwBuild& eb, cudaStream_t s, bool dry) {
  if (!eb.plan.in[0] || (F::kR1 && !eb.plan.in[1]) || (F::kR2 && !eb.plan.in[2]) ||
      (!eb.plan.out[0] && !eb.plan.out[1]))
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  if (eb.vec == 8) return launch_ew_kernel<F, 8, NOUT, bf16>(eb.plan, s);
  if (eb.vec == 4) return launch_ew_kernel<F, 4, NOUT, bf16>(eb.plan, s);
  return launch_ew_kernel<F, 1, NOUT, bf16>(eb.plan, s);
}

// GeLU by table: a flat plan, grid (at most one CTA per SM) in plan.n_cta.
template <bool BWD>
cudaError_t gelu_table_bf16(const EwBuild& eb, cudaStream_t s, bool dry) {
  const EwPlan& p = eb.plan;
  if (!p.flat || !p.in[0] || (BWD && !p.in[1]) || !p.out[0] || p.n_cta == 0 || p.n_cta > kSms)
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  constexpr size_t smem = GeluTab<BWD>::kSmemBytes;
  auto kern = eb.vec == 8 ? k_gelu_bf16<BWD, 8> : eb.vec == 4 ? k_gelu_bf16<BWD, 4> : k_gelu_bf16<BWD, 1>;
  kern = with_smem(kern, smem);
  if (!kern) return cudaErrorInvalidValue;
  return launch_k(kern, p.n_cta, kGeluTabThreads, smem, s, p);
}

template <int OP>
cudaError_t direct_bf16(int want, const EwBuild& eb, cudaStream_t s, bool dry) {
  switch (want) {
    case 1: return launch_ew_bf16<BwdDirectF<OP, 1, true>, 2>(eb, s, dry);
    case 2: return launch_ew_bf16<BwdDirectF<OP, 2, true>, 2>(eb, s, dry);
    default: return launch_ew_bf16<BwdDirectF<OP, 3, true>, 2>(eb, s, dry);
  }
}

template <int OP, int WHICH>
cudaError_t red_bf16(const RedBuild& rb, cudaStream_t s, bool dry) {
  const RedPlan& p = rb.plan;
  const bool has_d = p.d_out != nullptr;
  if (!p.g || (RedTerms<OP, WHICH>::reads_a(has_d) && !p.a) ||
      (RedTerms<OP, WHICH>::reads_b(has_d) && !p.b) || !p.x_final ||
      (p.nslots > 1 && !p.partial) || p.cluster > 1)
    return cudaErrorInvalidValue;
  // With partial slots, division's grad_b stores its factors after the slots:
  // only a plan whose workspace was sized for them may run.
  if (RedTerms<OP, WHICH>::kPost && p.nslots > 1 && !rb.comb.post) return cudaErrorInvalidValue;
  if (p.stages != 0 && (rb.vec * sizeof(bf16) != 16 || p.stages < 2 || p.stages > 3 ||
                        p.stage_ns < 1 || p.stage_ns > 2))
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  const size_t smem = red_smem_bytes(p, rb.vec, p.stages, p.stage_ns);
  cudaError_t e;
  if (p.inner_kept) {
    e = rb.vec == 8   ? launch_k(with_smem(k_reduce<OP, WHICH, 8, true, false, bf16>, smem), p.n_cta,
                                 kThreads, smem, s, p)
        : rb.vec == 4 ? launch_k(k_reduce<OP, WHICH, 4, true, false, bf16>, p.n_cta, kThreads, smem, s, p)
                      : launch_k(k_reduce<OP, WHICH, 1, true, false, bf16>, p.n_cta, kThreads, smem, s, p);
  } else {
    e = rb.vec == 8   ? launch_k(with_smem(k_reduce<OP, WHICH, 8, false, false, bf16>, smem), p.n_cta,
                                 kThreads, smem, s, p)
        : rb.vec == 4 ? launch_k(k_reduce<OP, WHICH, 4, false, false, bf16>, p.n_cta, kThreads, smem, s, p)
                      : launch_k(k_reduce<OP, WHICH, 1, false, false, bf16>, p.n_cta, kThreads, smem, s, p);
  }
  if (e != cudaSuccess || p.nslots <= 1) return e;
  return launch_combine_bf16(rb.comb, s);
}

template <int OP>
cudaError_t red_op_bf16(int which, const RedBuild& rb, cudaStream_t s, bool dry) {
  return which == 0 ? red_bf16<OP, 0>(rb, s, dry) : red_bf16<OP, 1>(rb, s, dry);
}

}  // namespace

cudaError_t launch_combine_bf16(CombinePlan c, cudaStream_t s) {
  combine_vectorize(&c);
  const unsigned nblk = static_cast<unsigned>(combine_blocks(c));
  return c.vec == 4 ? launch_k(k_combine<bf16, 4>, nblk, kThreads, 0, s, c)
                    : launch_k(k_combine<bf16, 1>, nblk, kThreads, 0, s, c);
}

cudaError_t launch_fwd_bf16(int op, const EwBuild& eb, cudaStream_t s, bool dry) {
  switch (op) {
    case OP_ADD: return launch_ew_bf16<FwdF<OP_ADD>, 1>(eb, s, dry);
    case OP_SUB: return launch_ew_bf16<FwdF<OP_SUB>, 1>(eb, s, dry);
    case OP_MUL: return launch_ew_bf16<FwdF<OP_MUL>, 1>(eb, s, dry);
    default:
      return eb.uni1 ? launch_ew_bf16<FwdF<OP_DIV, true, true>, 1>(eb, s, dry)
                     : launch_ew_bf16<FwdF<OP_DIV, true>, 1>(eb, s, dry);
  }
}

cudaError_t launch_unary_fwd_bf16(int uop, const EwBuild& eb, cudaStream_t s, bool dry) {
  if (uop == UN_GELU && eb.gelu_tab) return gelu_table_bf16<false>(eb, s, dry);
  return uop == UN_SCALE ? launch_ew_bf16<UnaryF<UN_SCALE>, 1>(eb, s, dry)
                         : launch_ew_bf16<UnaryF<UN_GELU, true>, 1>(eb, s, dry);
}

cudaError_t launch_unary_bwd_bf16(int uop, const EwBuild& eb, cudaStream_t s, bool dry) {
  if (uop == UN_GELU && eb.gelu_tab) return gelu_table_bf16<true>(eb, s, dry);
  return uop == UN_SCALE ? launch_ew_bf16<UnaryBwdF<UN_SCALE>, 1>(eb, s, dry)
                         : launch_ew_bf16<UnaryBwdF<UN_GELU, true>, 1>(eb, s, dry);
}

cudaError_t launch_bwd_direct_bf16(int op, int want, const EwBuild& eb, cudaStream_t s, bool dry) {
  switch (op) {
    case OP_ADD: return direct_bf16<OP_ADD>(want, eb, s, dry);
    case OP_SUB: return direct_bf16<OP_SUB>(want, eb, s, dry);
    case OP_MUL: return direct_bf16<OP_MUL>(want, eb, s, dry);
    default: return direct_bf16<OP_DIV>(want, eb, s, dry);
  }
}

cudaError_t occupancy_bf16(int which, int* planned, int* actual) {
  switch (which) {
    case 0:  // the flat kernel's 8-wide GeLU forward
      *planned = kOccGeluFwdWide;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_flat<UnaryF<UN_GELU, true>, 8, 1, bf16>, kThreads, 0);
    case 1:  // GeLU by table, forward and backward, 8-wide: one CTA per SM
    case 2: {
      *planned = 1;
      const bool bwd = which == 2;
      const size_t smem = bwd ? GeluTab<true>::kSmemBytes : GeluTab<false>::kSmemBytes;
      auto kern = with_smem(bwd ? k_gelu_bf16<true, 8> : k_gelu_bf16<false, 8>, smem);
      if (!kern) return cudaErrorInvalidValue;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, kern, kGeluTabThreads, smem);
    }
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_copy_bf16(const EwBuild& eb, cudaStream_t s, bool dry) {
  return launch_ew_bf16<CopyF, 1>(eb, s, dry);
}

cudaError_t launch_reduce_bf16(int op, int which, const RedBuild& rb, cudaStream_t s, bool dry) {
  if (which == 2) return red_bf16<OP_ADD, 2>(rb, s, dry);
  switch (op) {
    case OP_ADD: return red_op_bf16<OP_ADD>(which, rb, s, dry);
    case OP_SUB: return red_op_bf16<OP_SUB>(which, rb, s, dry);
    case OP_MUL: return red_op_bf16<OP_MUL>(which, rb, s, dry);
    default: return red_op_bf16<OP_DIV>(which, rb, s, dry);
  }
}

namespace {
// One CTA per x bit pattern, threads stride over the y patterns.  out[0],
// out[1]: quot_short against the IEEE divide (binary32 bits); out[2],
// out[3]: quot_bf16 against the IEEE divide, both rounded to bfloat16.
__global__ void __launch_bounds__(kThreads) k_div_short_check(unsigned long long* out) {
  const uint32_t xb = blockIdx.x;
  const float x = __uint_as_float(xb << 16);
  uint32_t bad[2] = {0, 0}, first[2] = {0xffffffffu, 0xffffffffu};
  for (uint32_t yb = threadIdx.x; yb < 65536u; yb += blockDim.x) {
    const float y = __uint_as_float(yb << 16);
    Vec<1> xv, yv, q1, q2;
    xv.v[0] = x;
    yv.v[0] = y;
    quot_short(xv, yv, q1);
    quot_bf16(xv, yv, q2);
    const float r = __fdiv_rn(x, y);
    const uint32_t key = (xb << 16) | yb;
    const float a = q1.v[0];
    if (!(__float_as_uint(a) == __float_as_uint(r) || (a != a && r != r))) {
      ++bad[0];
      first[0] = key < first[0] ? key : first[0];
    }
    const float b16 = __bfloat162float(__float2bfloat16_rn(q2.v[0]));
    const float r16 = __bfloat162float(__float2bfloat16_rn(r));
    if (!(__float_as_uint(b16) == __float_as_uint(r16) || (b16 != b16 && r16 != r16))) {
      ++bad[1];
      first[1] = key < first[1] ? key : first[1];
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t n = __reduce_add_sync(0xffffffffu, bad[k]);
    const uint32_t f = __reduce_min_sync(0xffffffffu, first[k]);
    if ((threadIdx.x & 31u) == 0 && n) {
      atomicAdd(out + 2 * k, static_cast<unsigned long long>(n));
      atomicMin(out + 2 * k + 1, static_cast<unsigned long long>(f));
    }
  }
}
}  // namespace

cudaError_t launch_div_short_check(unsigned long long* out, cudaStream_t s) {
  k_div_short_check<<<65536, kThreads, 0, s>>>(out);
  return cudaGetLastError();
}

}  // namespace zr
