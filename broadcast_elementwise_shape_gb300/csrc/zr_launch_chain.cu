// zr_launch_chain.cu — instantiations and launches of the two-op chain
// kernels: the forward (k_elementwise with ChainF) and the fused backward
// (k_chain_bwd and its second passes).
#include "zr_launch.h"
#include "zr_chain.cuh"

namespace zr {

namespace {

template <int OP1, int OP2, bool C_ONE>
cudaError_t launch_chain_fwd_c(const EwBuild& eb, cudaStream_t s) {
  using F = ChainF<OP1, OP2, C_ONE>;
  if (eb.vec == 4) return launch_ew_kernel<F, 4, 1>(eb.plan, s);
  return launch_ew_kernel<F, 1, 1>(eb.plan, s);
}

// c_one: c has one element (read once per thread).
struct FwdArg {
  const EwBuild& eb;
  bool c_one;
};
template <int OP1, int OP2>
cudaError_t launch_chain_fwd_t(const FwdArg& f, cudaStream_t s) {
  return f.c_one ? launch_chain_fwd_c<OP1, OP2, true>(f.eb, s)
                 : launch_chain_fwd_c<OP1, OP2, false>(f.eb, s);
}


template <int OP1, int OP2>
cudaError_t launch_chain_bwd_t(const ChainBuild& cb, cudaStream_t s) {
  const ChainPlan& cp = cb.plan;
  const RedPlan& p = cp.r;
  const uint32_t table_rows = p.rows_per_blk < kMaxTileRows ? p.rows_per_blk : kMaxTileRows;
  const size_t smem = size_t(table_rows) * kMaxOperands * sizeof(int64_t) + size_t(kThreads) * 4 * sizeof(float);
  cudaError_t e = cp.c_scalar ? launch_k(k_chain_bwd<OP1, OP2, true>, p.n_cta, kThreads, smem, s, cp)
                              : launch_k(k_chain_bwd<OP1, OP2, false>, p.n_cta, kThreads, smem, s, cp);
  if (e != cudaSuccess) return e;
  // With c shaped like b, one second pass finishes grad_b and grad_c.
  if (p.nslots > 1) e = launch_combine_f32(cb.comb_b, s);
  if (e == cudaSuccess && cp.c_scalar && p.n_cta > 1) e = launch_combine_f32(cb.comb_c, s);
  return e;
}

#define ZR_CHAIN_CASES(OP1, FN, ARG)                         \
  switch (op2) {                                             \
    case OP_ADD: return FN<OP1, OP_ADD>(ARG, s);             \
    case OP_SUB: return FN<OP1, OP_SUB>(ARG, s);             \
    case OP_MUL: return FN<OP1, OP_MUL>(ARG, s);             \
    default: return FN<OP1, OP_DIV>(ARG, s);                 \
  }

cudaError_t fwd_dispatch(int op1, int op2, const FwdArg& f, cudaStream_t s) {
  switch (op1) {
    case OP_ADD: ZR_CHAIN_CASES(OP_ADD, launch_chain_fwd_t, f)
    case OP_SUB: ZR_CHAIN_CASES(OP_SUB, launch_chain_fwd_t, f)
    case OP_MUL: ZR_CHAIN_CASES(OP_MUL, launch_chain_fwd_t, f)
    default: ZR_CHAIN_CASES(OP_DIV, launch_chain_fwd_t, f)
  }
}

cudaError_t bwd_dispatch(int op1, int op2, const ChainBuild& cb, cudaStream_t s) {
  switch (op1) {
    case OP_ADD: ZR_CHAIN_CASES(OP_ADD, launch_chain_bwd_t, cb)
    case OP_SUB: ZR_CHAIN_CASES(OP_SUB, launch_chain_bwd_t, cb)
    case OP_MUL: ZR_CHAIN_CASES(OP_MUL, launch_chain_bwd_t, cb)
    default: ZR_CHAIN_CASES(OP_DIV, launch_chain_bwd_t, cb)
  }
}
#undef ZR_CHAIN_CASES

}  // namespace

cudaError_t launch_chain_fwd(int op1, int op2, bool c_one, const EwBuild& eb, cudaStream_t s,
                             bool dry) {
  if (!eb.plan.in[0] || !eb.plan.in[1] || !eb.plan.in[2] || !eb.plan.out[0])
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  return fwd_dispatch(op1, op2, FwdArg{eb, c_one}, s);
}

cudaError_t launch_chain_bwd(int op1, int op2, const ChainBuild& cb, cudaStream_t s, bool dry) {
  const ChainPlan& cp = cb.plan;
  const RedPlan& p = cp.r;
  // The kernel dereferences every one of these.
  if (!p.g || !p.a || !p.b || !cp.c || !p.d_out || !p.x_final || !cp.c_final ||
      !p.inner_kept || p.cluster > 1 || (p.nslots > 1 && !p.partial) ||
      (!cp.c_scalar && p.nslots > 1 && (cb.comb_b.split != p.nout || !cb.comb_b.out2)) ||
      (cp.c_scalar && p.n_cta > 1 && !cp.c_partial))
    return cudaErrorInvalidValue;
  // With a division in the chain the kernel stores per-output factors after
  // the partial slots: only a plan whose workspace holds them may run.
  const bool rows_post = op1 == OP_DIV || (!cp.c_scalar && op2 == OP_DIV);
  if ((rows_post && p.nslots > 1 && !cb.comb_b.post) ||
      (cp.c_scalar && op2 == OP_DIV && p.n_cta > 1 && !cb.comb_c.post))
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  return bwd_dispatch(op1, op2, cb, s);
}

cudaError_t occupancy_chain(int which, int* planned, int* actual) {
  const size_t smem = size_t(kMaxTileRows) * kMaxOperands * sizeof(int64_t) +
                      size_t(kThreads) * 4 * sizeof(float);
  switch (which) {
    case 0:
      *planned = kOccEwBwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_elementwise<ChainF<OP_MUL, OP_ADD, false>, 4, 1>, kThreads,
          size_t(kMaxTileRows) * kMaxOperands * sizeof(int64_t));
    case 3:
      *planned = kOccEwFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_elementwise<ChainF<OP_ADD, OP_DIV, true>, 4, 1>, kThreads,
          size_t(kMaxTileRows) * kMaxOperands * sizeof(int64_t));
    case 1:
      *planned = kOccChain;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_chain_bwd<OP_MUL, OP_ADD, false>, kThreads, smem);
    case 2:
      *planned = kOccChain;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_chain_bwd<OP_ADD, OP_DIV, true>, kThreads, smem);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zr
